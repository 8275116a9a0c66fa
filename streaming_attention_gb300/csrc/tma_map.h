// Host-side TMA tensor-map encoding (the driver entry point is looked up once
// through the runtime, so the library does not link the driver directly).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace attn {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A [heads][rows][D] tensor of 16-bit (elem_bytes 2, BF16 or FP16) or 8-bit
// (elem_bytes 1, read as raw bytes) elements, read in boxes of 128 bytes along
// D x box_rows x 1 with the 128-byte swizzle. Out-of-range elements read 0.
inline bool make_tensor_map(CUtensorMap* m, const void* base, int D, int rows, int heads, int box_rows, bool bf16,
                            int elem_bytes = 2) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t eb = (cuuint64_t)elem_bytes;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)rows * D * eb};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType ty = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : bf16          ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = fn(m, ty, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace attn
