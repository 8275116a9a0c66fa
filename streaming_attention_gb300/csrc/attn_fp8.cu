// C ABI of the forward pass on E4M3 inputs: metadata validation, the empty
// and key-less cases, and the tcgen05 prefill kernel in its 8-bit form.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

__global__ void fill_f32_kernel(float* x, int64_t n, float value) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        x[i] = value;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int M, int N, int D, int causal, int window, float scale, float q_descale,
                            float k_descale, float v_descale, int out_dtype, void* stream) {
    Problem p;
    // the 16-bit validation covers sizes, GQA, element counts, pointers and
    // alignment; the element count of an 8-bit tensor is the same bound
    int rc = validate_problem(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, out_dtype, &p);
    if (rc != ATTN_OK) return rc;
    if (D != 128) return ATTN_ERR_HEADDIM;
    const int64_t rows = (int64_t)B * Hq * M;
    if (rows > 0 && lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ALIGN;
    if (rows == 0) return ATTN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {  // no keys: output 0, log-sum-exp -inf
        cudaError_t e = cudaMemsetAsync(o, 0, (size_t)rows * D * 2, s);
        if (e == cudaSuccess && lse) {
            const int blocks = (int)((rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024);
            fill_f32_kernel<<<blocks, 256, 0, s>>>(lse, rows, -INFINITY);
            e = cudaGetLastError();
        }
        return cuda_status(e);
    }
    int* status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    p.lse = lse;
    // logits of the dequantized tensors: scale * q_descale * k_descale * <q, k>
    p.scale_log2 = (float)((double)p.scale * (double)q_descale * (double)k_descale * (double)kLog2e);
    if (!prefill_supported(p)) return ATTN_ERR_PATH;
    return launch_prefill_e4m3(p, q, k, v, o, status, v_descale, s);
}
