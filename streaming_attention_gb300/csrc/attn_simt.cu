// CUDA-core streaming attention: the general path for every supported head
// dimension (16, 32, 64, 128), any ragged M/N, causal and window masks, GQA,
// and key-range splits. One warp owns one query row and carries its running
// (m, l, acc) across tiles of 32 keys, never holding more than one tile of
// scores ("Compare reasoning after your own attempt", central-idea table, A3
// row). Keys and values of a tile are staged once in shared memory for the
// four rows of the block.
//
// Also holds the merge kernel that combines split summaries with the
// common-maximum rule (same table, A1 row).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kRowsPerBlock = 4;  // one warp per query row
constexpr int kKeyTile = 32;      // one key per lane per tile

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

struct SimtArgs {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* ws_m;
    float* ws_l;
    float* ws_acc;
    int B, Hq, Hkv, M, N, G;
    int causal, window;
    float scale_log2;
    int klo, khi, kbase, chunk, S;  // splits: [kbase + z*chunk, +chunk) within [klo, khi)
    int partial;  // 1: write (m, l, acc) summaries; 0: write normalized o
    float* lse;   // optional per-row log-sum-exp (natural log) when writing o
};

template <typename T, int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32) attn_simt_kernel(SimtArgs a) {
    constexpr int EPL = (D + 31) / 32;  // output elements per lane
    __shared__ float qs[kRowsPerBlock][D];
    __shared__ float ks[kKeyTile][D + 1];  // +1: lane-per-key reads hit distinct banks
    __shared__ float vs[kKeyTile][D];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y;
    const int b = bh / a.Hq, h = bh % a.Hq, g = h / a.G;
    const int i0 = blockIdx.x * kRowsPerBlock;
    const int i = i0 + warp;
    const int off = a.N - a.M;  // position of row i is i + off
    const T* Q = reinterpret_cast<const T*>(a.q) + ((size_t)bh * a.M) * D;
    const T* K = reinterpret_cast<const T*>(a.k) + ((size_t)(b * a.Hkv + g) * a.N) * D;
    const T* V = reinterpret_cast<const T*>(a.v) + ((size_t)(b * a.Hkv + g) * a.N) * D;

    // keys visible to any row of this block, within this split (both bounds
    // of a row's range grow with its position)
    const int i_last = min(i0 + kRowsPerBlock - 1, a.M - 1);
    int lo_first, hi_first, lo_last, hi_last;
    key_range(i0 + off, a.N, a.causal, a.window, &lo_first, &hi_first);
    key_range(i_last + off, a.N, a.causal, a.window, &lo_last, &hi_last);
    const int s_lo = a.kbase + blockIdx.z * a.chunk;
    const int s_hi = min(s_lo + a.chunk, a.khi);
    const int lo = max(lo_first, s_lo);
    const int hi = min(hi_last, s_hi);

    // this row's own visible range
    int r_lo = 0, r_hi = 0;
    if (i < a.M) key_range(i + off, a.N, a.causal, a.window, &r_lo, &r_hi);

    for (int d = threadIdx.x; d < kRowsPerBlock * D; d += blockDim.x) {
        int r = d / D, c = d % D;
        qs[r][c] = (i0 + r < a.M) ? to_f32(Q[(size_t)(i0 + r) * D + c]) : 0.f;
    }

    float m = -INFINITY, l = 0.f;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;

    for (int j0 = lo; j0 < hi; j0 += kKeyTile) {
        __syncthreads();  // previous tile fully consumed (and qs written)
        for (int x = threadIdx.x; x < kKeyTile * D; x += blockDim.x) {
            int r = x / D, c = x % D;
            int j = j0 + r;
            bool in = j < hi;
            ks[r][c] = in ? to_f32(K[(size_t)j * D + c]) : 0.f;
            vs[r][c] = in ? to_f32(V[(size_t)j * D + c]) : 0.f;
        }
        __syncthreads();
        if (i < a.M) {
            const int j = j0 + lane;
            float t = -INFINITY;  // masked and padded keys score -inf
            if (j < hi && j >= r_lo && j < r_hi) {
                float dot = 0.f;
#pragma unroll 8
                for (int d = 0; d < D; ++d) dot = fmaf(qs[warp][d], ks[lane][d], dot);
                t = dot * a.scale_log2;
            }
            const float m_new = fmaxf(m, warp_max(t));
            // ghost-row pin: while every key so far is masked, use 0 as the max
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = exp2f(m - m_use);
            const float p = exp2f(t - m_use);
            l = l * alpha + warp_sum(p);
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
#pragma unroll 4
            for (int jj = 0; jj < kKeyTile; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const int d = lane + 32 * e;
                    if (d < D) acc[e] = fmaf(pj, vs[jj][d], acc[e]);
                }
            }
            m = m_new;
        }
    }

    if (i >= a.M) return;
    const size_t row = (size_t)bh * a.M + i;
    if (a.partial) {
        const size_t slot = row * a.S + blockIdx.z;
        if (lane == 0) {
            a.ws_m[slot] = m;
            a.ws_l[slot] = l;
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int d = lane + 32 * e;
            if (d < D) a.ws_acc[slot * D + d] = acc[e];
        }
    } else {
        const float inv = l > 0.f ? 1.f / l : 0.f;  // no visible key: output 0
        // log sum_j e^(scale s_j) = ln 2 * (m + log2 l); -inf for a row with no key
        if (a.lse && lane == 0) a.lse[row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        T* O = reinterpret_cast<T*>(a.o) + row * D;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int d = lane + 32 * e;
            if (d < D) O[d] = from_f32<T>(acc[e] * inv);
        }
    }
}

// Merge of S summaries, one thread per output element (row, d): every load is
// independent of the arithmetic, so the whole merge is one memory round trip.
// unit converts the stored maxima to base 2 (1 for base-2 maxima, log2(e) for
// natural-log maxima); out_scale multiplies the merged output (a V
// dequantization factor; 1 otherwise).
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads)
    attn_merge_kernel(const float* __restrict__ m, const float* __restrict__ l, const float* __restrict__ acc,
                      void* o, float* m_out, float* l_out, float* lse_out, int rows, int S, int D, int out_dtype,
                      float unit, int programmatic, float out_scale) {
    // A programmatically launched successor (the next decode split grid) may start
    // its setup now; it waits for this grid's completion before touching memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (programmatic) asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t idx = (size_t)blockIdx.x * kMergeThreads + threadIdx.x;
    const size_t row = idx / D;
    const int d = (int)(idx % D);
    if (row >= (size_t)rows) return;
    const float* mr = m + row * S;
    const float* lr = l + row * S;
    const float* ar = acc + row * S * D + d;

    float mx = -INFINITY;
#pragma unroll 8
    for (int s = 0; s < S; ++s) mx = fmaxf(mx, mr[s]);
    float L = 0.f, x = 0.f;
#pragma unroll 8
    for (int s = 0; s < S; ++s) {
        const float ms = mr[s];
        // an empty summary (m = -inf) weighs 0; never forms -inf - (-inf)
        const float ws = (ms == -INFINITY) ? 0.f : exp2f((ms - mx) * unit);
        L = fmaf(ws, lr[s], L);
        x = fmaf(ws, ar[(size_t)s * D], x);
    }
    x *= L > 0.f ? out_scale / L : 0.f;
    const size_t out = row * D + d;
    if (out_dtype == ATTN_BF16)
        reinterpret_cast<__nv_bfloat16*>(o)[out] = __float2bfloat16_rn(x);
    else if (out_dtype == ATTN_FP16)
        reinterpret_cast<__half*>(o)[out] = __float2half_rn(x);
    else
        reinterpret_cast<float*>(o)[out] = x;
    if (d == 0) {
        if (m_out) m_out[row] = mx;
        if (l_out) l_out[row] = L;
        // the merged log-sum-exp in natural log: mx * unit is the base-2 maximum
        if (lse_out) lse_out[row] = L > 0.f ? (mx * unit + log2f(L)) * kLn2 : -INFINITY;
    }
}

template <typename T, int D>
cudaError_t launch_simt_t(const SimtArgs& a, cudaStream_t stream) {
    dim3 grid((a.M + kRowsPerBlock - 1) / kRowsPerBlock, a.B * a.Hq, a.S);
    attn_simt_kernel<T, D><<<grid, kRowsPerBlock * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_simt_d(const SimtArgs& a, int D, cudaStream_t stream) {
    switch (D) {
        case 16: return launch_simt_t<T, 16>(a, stream);
        case 32: return launch_simt_t<T, 32>(a, stream);
        case 64: return launch_simt_t<T, 64>(a, stream);
        case 128: return launch_simt_t<T, 128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_simt(const Problem& p, const void* q, const void* k, const void* v, void* o, int chunk,
                        int S, const SplitWorkspace* ws, cudaStream_t stream) {
    SimtArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.ws_m = ws ? ws->m : nullptr;
    a.ws_l = ws ? ws->l : nullptr;
    a.ws_acc = ws ? ws->acc : nullptr;
    a.B = p.B;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.M = p.M;
    a.N = p.N;
    a.G = p.G;
    a.causal = p.causal;
    a.window = p.window;
    a.scale_log2 = p.scale_log2;
    a.klo = ws ? p.klo : 0;
    a.khi = ws ? p.khi : p.N;
    a.kbase = ws ? split_base(p) : 0;
    a.chunk = ws ? chunk : (p.N > 0 ? p.N : 1);
    a.S = ws ? S : 1;
    a.partial = ws ? 1 : 0;
    a.lse = ws ? nullptr : p.lse;
    if (p.dtype == ATTN_BF16) return launch_simt_d<__nv_bfloat16>(a, p.D, stream);
    return launch_simt_d<__half>(a, p.D, stream);
}

cudaError_t launch_merge(const float* m, const float* l, const float* acc, void* o, float* m_out, float* l_out,
                         float* lse_out, int rows, int S, int D, int out_dtype, float unit, bool programmatic,
                         cudaStream_t stream, float out_scale) {
    if (rows == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(((size_t)rows * D + kMergeThreads - 1) / kMergeThreads));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_merge_kernel, m, l, acc, o, m_out, l_out, lse_out, rows, S, D, out_dtype,
                              unit, programmatic ? 1 : 0, out_scale);
}

}  // namespace attn
