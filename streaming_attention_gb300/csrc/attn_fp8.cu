// C ABI of attention on E4M3 inputs: metadata validation, the empty and
// key-less cases, the path choice, and the tcgen05 prefill and split-KV decode
// kernels in their 8-bit forms (the decode's summaries merge with the V
// dequantization factor applied). Paged decode on an E4M3 cache is in
// attn_paged.cu.
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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// AUTO: the split-KV decode for few grouped rows over a long key range (the
// rule of the 16-bit forward), else the prefill kernel
int choose_fp8_path(const Problem& p, int path) {
    if (path != ATTN_PATH_AUTO) return path;
    if (p.D == 128 && decode_tc_supported(p) && (int64_t)p.G * p.M <= 16 && (p.khi - p.klo) >= 512)
        return ATTN_PATH_DECODE;
    return ATTN_PATH_PREFILL;
}

int run_decode(const Problem& p, const void* q, const void* k, const void* v, void* o, float v_descale, void* ws,
               size_t ws_bytes, int* status, cudaStream_t s) {
    int chunk = 0, S = 0;
    decode_plan_tc(p, &chunk, &S, true);
    const int rows = p.B * p.Hq * p.M;
    if (!ws || ws_bytes < split_workspace_bytes(rows, S, p.D)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(ws)) return ATTN_ERR_ALIGN;
    SplitWorkspace w = split_workspace(ws, rows, S, p.D);
    DecodeOut out{o, p.lse, v_descale, false};
    if (launch_decode_e4m3(p, q, k, v, chunk, S, w, status, s, &out) != cudaSuccess) return ATTN_ERR_CUDA;
    if (out.merged) return ATTN_OK;
    return cuda_status(
        launch_merge(w.m, w.l, w.acc, o, nullptr, nullptr, p.lse, rows, S, p.D, p.dtype, 1.0f, true, s, v_descale));
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" size_t attn_fwd_fp8_workspace_bytes(int B, int Hq, int Hkv, int M, int N, int D, int causal, int window,
                                               int path) {
    static const int16_t dummy[8] __attribute__((aligned(16))) = {};
    Problem p;
    if (path < ATTN_PATH_AUTO || path > ATTN_PATH_DECODE || path == ATTN_PATH_SIMT) return 0;
    if (validate_problem(dummy, dummy, dummy, dummy, B, Hq, Hkv, M, N, D, causal, window, 0.f, ATTN_BF16, &p) !=
            ATTN_OK ||
        D != 128)
        return 0;  // D = 64 runs the prefill kernel, which needs no workspace
    if ((int64_t)B * Hq * M == 0 || N == 0) return 0;
    if (choose_fp8_path(p, path) != ATTN_PATH_DECODE || !decode_tc_supported(p)) return 0;
    int chunk = 0, S = 0;
    decode_plan_tc(p, &chunk, &S, true);
    return split_workspace_bytes(p.B * p.Hq * p.M, S, p.D);
}

extern "C" int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int M, int N, int D, int causal, int window, float scale, float q_descale,
                            float k_descale, float v_descale, attn_dtype_t out_dtype, int path, void* workspace,
                            size_t ws_bytes, void* stream) {
    if (path < ATTN_PATH_AUTO || path > ATTN_PATH_DECODE || path == ATTN_PATH_SIMT) return ATTN_ERR_PATH;
    Problem p;
    // the 16-bit validation covers sizes, GQA, element counts, pointers and
    // alignment; the element count of an 8-bit tensor is the same bound
    int rc = validate_problem(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, out_dtype, &p);
    if (rc != ATTN_OK) return rc;
    if (D != 128 && D != 64) return ATTN_ERR_HEADDIM;
    const int64_t rows = (int64_t)B * Hq * M;
    if (rows > 0 && lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ALIGN;
    path = choose_fp8_path(p, path);
    if (path == ATTN_PATH_DECODE && (D != 128 || !decode_tc_supported(p))) return ATTN_ERR_PATH;
    if (path == ATTN_PATH_PREFILL && !prefill_supported(p)) return ATTN_ERR_PATH;
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
    if (path == ATTN_PATH_PREFILL) return launch_prefill_e4m3(p, q, k, v, o, status, v_descale, s);
    if (workspace) return run_decode(p, q, k, v, o, v_descale, workspace, ws_bytes, status, s);
    int chunk = 0, S = 0;
    decode_plan_tc(p, &chunk, &S, true);
    const size_t bytes = split_workspace_bytes(p.B * p.Hq * p.M, S, p.D);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = run_decode(p, q, k, v, o, v_descale, ws, bytes, status, s);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}
