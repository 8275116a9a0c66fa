// C ABI of split-KV decode over a paged KV cache (16-bit or E4M3): metadata
// validation, the split plan, and the kernels: the tcgen05 split kernel in
// paged mode (D = 128; D = 64 for 16-bit caches) or the grouped CUDA-core
// kernel (every other head dimension), then the merge kernel.
// Attention over a KV-cache slice is the decode step the course's plan names
// next ("Kernel Notes & Checklist", section 3, the plan, week +3: sliding
// window + GQA + KV-cache slice); pages of the cache are gathered by the TMA
// producer through the block table, so no copy of the cache is ever made.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

constexpr int64_t kI32Max = 2147483647LL;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool page_size_ok(int ps) { return ps == 16 || ps == 32 || ps == 64 || (ps > 0 && ps % 128 == 0); }

struct PagedCall {
    Problem p;
    PagedKV kv;
};

// Metadata only (never values): shapes, head dimension, group size, 32-bit
// element counts, null pointers of non-empty tensors, alignment.
int validate_paged(const void* q, const void* kp, const void* vp, const int* table, const int* lens, const void* o,
                   int B, int Hq, int Hkv, int M, int D, int num_pages, int page_size, int max_pages,
                   int max_seq_len, int causal, int window, float scale, int dtype, PagedCall* c,
                   bool e4m3 = false) {
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
    if (B < 0 || Hq < 0 || Hkv < 0 || M < 0 || D <= 0 || num_pages < 0 || max_pages < 0 || max_seq_len < 0)
        return ATTN_ERR_SHAPE;
    if (Hq > 0 && Hkv == 0) return ATTN_ERR_SHAPE;
    if (!page_size_ok(page_size)) return ATTN_ERR_SHAPE;
    if (Hq > 0 && Hq % Hkv != 0) return ATTN_ERR_GQA;
    if (D != 16 && D != 32 && D != 64 && D != 128) return ATTN_ERR_HEADDIM;
    const int G = Hkv > 0 ? Hq / Hkv : 1;
    const int64_t nq = (int64_t)B * Hq * M * D;
    const int64_t npool = (int64_t)num_pages * Hkv * page_size * D;
    const int64_t ntab = (int64_t)B * max_pages;
    if (nq > kI32Max || npool > kI32Max || ntab > kI32Max || (int64_t)B * Hkv > 65535) return ATTN_ERR_OVERFLOW;
    if ((nq > 0 && (!q || !o)) || (npool > 0 && (!kp || !vp)) || (ntab > 0 && !table) || (B > 0 && !lens))
        return ATTN_ERR_NULL;
    if ((q && !aligned(q, 16)) || (o && !aligned(o, 16)) || (kp && !aligned(kp, 16)) || (vp && !aligned(vp, 16)) ||
        (table && !aligned(table, 4)) || (lens && !aligned(lens, 4)))
        return ATTN_ERR_ALIGN;
    const int64_t cover = (int64_t)max_pages * page_size;
    const int max_len = (int)(cover < max_seq_len ? cover : max_seq_len);
    Problem& p = c->p;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.M = M;
    p.N = max_len;
    p.D = D;
    p.causal = causal ? 1 : 0;
    p.window = window > 0 ? window : 0;
    p.scale = (scale == 0.0f) ? (float)(1.0 / sqrt((double)D)) : scale;
    p.scale_log2 = p.scale * kLog2e;
    p.dtype = dtype;
    p.G = G;
    p.klo = 0;  // per sequence, in the kernel
    p.khi = max_len;
    p.lse = nullptr;
    c->kv = PagedKV{kp, vp, table, lens, num_pages, page_size, max_pages, max_len};
    if (!paged_tc_supported(p, e4m3) && !paged_group_supported(p)) return ATTN_ERR_OVERFLOW;
    return ATTN_OK;
}

bool nothing_to_attend(const PagedCall& c) { return c.kv.max_len == 0 || c.kv.num_pages == 0 || c.p.Hkv == 0; }

// The split plan of the kernel that runs this call.
void paged_plan(const PagedCall& c, bool e4m3, int* chunk, int* S) {
    if (paged_tc_supported(c.p, e4m3))
        decode_plan_paged(c.p, c.kv, chunk, S, e4m3);
    else
        paged_group_plan(c.p, c.kv, chunk, S);
}

// Scratch for the splits' summaries; the grouped kernel with one split writes
// the output itself and needs none.
size_t paged_workspace(const PagedCall& c, bool e4m3 = false) {
    int chunk = 0, S = 0;
    paged_plan(c, e4m3, &chunk, &S);
    if (!paged_tc_supported(c.p, e4m3) && S == 1) return 0;
    return split_workspace_bytes(c.p.B * c.p.Hq * c.p.M, S, c.p.D);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

int run_paged(const PagedCall& c, const void* q, void* o, void* ws, size_t ws_bytes, cudaStream_t stream,
              bool e4m3 = false, float v_descale = 1.0f) {
    const Problem& p = c.p;
    int chunk = 0, S = 0;
    paged_plan(c, e4m3, &chunk, &S);
    const int rows = p.B * p.Hq * p.M;
    if (!paged_tc_supported(p, e4m3)) {
        if (S == 1) return cuda_status(launch_paged_group(p, q, c.kv, chunk, S, nullptr, o, v_descale, e4m3, stream));
        if (!ws || ws_bytes < split_workspace_bytes(rows, S, p.D)) return ATTN_ERR_WORKSPACE;
        if (!aligned(ws, 16)) return ATTN_ERR_ALIGN;
        SplitWorkspace w = split_workspace(ws, rows, S, p.D);
        if (launch_paged_group(p, q, c.kv, chunk, S, &w, o, v_descale, e4m3, stream) != cudaSuccess)
            return ATTN_ERR_CUDA;
        return cuda_status(launch_merge(w.m, w.l, w.acc, o, nullptr, nullptr, nullptr, rows, S, p.D, p.dtype, 1.0f,
                                        false, stream, v_descale));
    }
    if (!ws || ws_bytes < split_workspace_bytes(rows, S, p.D)) return ATTN_ERR_WORKSPACE;
    if (!aligned(ws, 16)) return ATTN_ERR_ALIGN;
    int* status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    SplitWorkspace w = split_workspace(ws, rows, S, p.D);
    DecodeOut out{o, nullptr, v_descale, false};
    if (launch_decode_paged(p, q, c.kv, chunk, S, w, status, stream, &out, e4m3) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (out.merged) return ATTN_OK;
    return cuda_status(launch_merge(w.m, w.l, w.acc, o, nullptr, nullptr, nullptr, rows, S, p.D, p.dtype, 1.0f, true,
                                    stream, v_descale));
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

size_t attn_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int M, int D, int page_size, int max_pages,
                                         int max_seq_len, int causal, int window) {
    static const int16_t dummy[8] __attribute__((aligned(16))) = {};
    const int* idummy = reinterpret_cast<const int*>(dummy);
    PagedCall c;
    if (validate_paged(dummy, dummy, dummy, idummy, idummy, dummy, B, Hq, Hkv, M, D, 1, page_size, max_pages,
                       max_seq_len, causal, window, 0.f, ATTN_BF16, &c) != ATTN_OK)
        return 0;
    if ((int64_t)B * Hq * M == 0 || nothing_to_attend(c)) return 0;
    return paged_workspace(c);
}

int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                      const int* seq_lens, void* o, int B, int Hq, int Hkv, int M, int D, int num_pages,
                      int page_size, int max_pages, int max_seq_len, int causal, int window, float scale, attn_dtype_t dtype,
                      void* workspace, size_t ws_bytes, void* stream) {
    PagedCall c;
    int rc = validate_paged(q, k_pages, v_pages, block_table, seq_lens, o, B, Hq, Hkv, M, D, num_pages, page_size,
                            max_pages, max_seq_len, causal, window, scale, dtype, &c);
    if (rc != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((int64_t)B * Hq * M == 0) return ATTN_OK;
    if (nothing_to_attend(c))  // no sequence can hold a key: every row outputs 0
        return cuda_status(cudaMemsetAsync(o, 0, (size_t)B * Hq * M * D * 2, s));
    if (workspace) return run_paged(c, q, o, workspace, ws_bytes, s);
    const size_t bytes = paged_workspace(c);
    if (bytes == 0) return run_paged(c, q, o, nullptr, 0, s);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = run_paged(c, q, o, ws, bytes, s);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}

size_t attn_decode_paged_fp8_workspace_bytes(int B, int Hq, int Hkv, int M, int D, int page_size, int max_pages,
                                             int max_seq_len, int causal, int window) {
    static const int16_t dummy[8] __attribute__((aligned(16))) = {};
    const int* idummy = reinterpret_cast<const int*>(dummy);
    PagedCall c;
    if (validate_paged(dummy, dummy, dummy, idummy, idummy, dummy, B, Hq, Hkv, M, D, 1, page_size, max_pages,
                       max_seq_len, causal, window, 0.f, ATTN_BF16, &c, true) != ATTN_OK)
        return 0;
    if ((int64_t)B * Hq * M == 0 || nothing_to_attend(c)) return 0;
    return paged_workspace(c, true);
}

int attn_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                          const int* seq_lens, void* o, int B, int Hq, int Hkv, int M, int D, int num_pages,
                          int page_size, int max_pages, int max_seq_len, int causal, int window, float scale,
                          float q_descale, float k_descale, float v_descale, attn_dtype_t out_dtype, void* workspace,
                          size_t ws_bytes, void* stream) {
    PagedCall c;
    int rc = validate_paged(q, k_pages, v_pages, block_table, seq_lens, o, B, Hq, Hkv, M, D, num_pages, page_size,
                            max_pages, max_seq_len, causal, window, scale, out_dtype, &c, true);
    if (rc != ATTN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((int64_t)B * Hq * M == 0) return ATTN_OK;
    if (nothing_to_attend(c)) return cuda_status(cudaMemsetAsync(o, 0, (size_t)B * Hq * M * D * 2, s));
    // logits of the dequantized tensors: scale * q_descale * k_descale * <q, k>
    c.p.scale_log2 = (float)((double)c.p.scale * (double)q_descale * (double)k_descale * (double)kLog2e);
    if (workspace) return run_paged(c, q, o, workspace, ws_bytes, s, true, v_descale);
    const size_t bytes = paged_workspace(c, true);
    if (bytes == 0) return run_paged(c, q, o, nullptr, 0, s, true, v_descale);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = run_paged(c, q, o, ws, bytes, s, true, v_descale);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}

}  // extern "C"
