// Grouped CUDA-core decode over a paged KV cache: the head dimensions the
// tcgen05 split kernel does not take (16 and 32; 64 for E4M3 caches), for
// 16-bit and E4M3 caches.
//
// One block owns one split of one sequence's key range for one KV head and up
// to eight of that head's grouped query rows (one warp per row: query head
// h = g*G + r / M, row i = r % M). Each 32-key tile is gathered from its pages
// once, through the block table, into shared memory and read there by all the
// block's rows, so a KV head's keys leave HBM once per split and row chunk, not
// once per query head. Each row carries its running (m, l, acc) across tiles
// and never holds more than one tile of scores ("Compare reasoning after your
// own attempt", central-idea table, A3 row); the splits' summaries are combined
// by the common-maximum merge (same table, A1 row). The decode step over a
// KV-cache slice is the one the course's plan names next ("Kernel Notes &
// Checklist", section 3, the plan, week +3).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kGWarps = 8;   // grouped rows per block, one warp each
constexpr int kGKeys = 32;   // keys per staged tile, one per lane
constexpr int kGTile = 128;  // split granularity in keys

struct E4M3In {};  // tag: 8-bit E4M3 inputs

struct GroupArgs {
    const void* q;
    const void* kp;
    const void* vp;
    const int* table;
    const int* lens;
    void* o;  // written directly when S == 1
    float* ws_m;
    float* ws_l;
    float* ws_acc;
    int Hq, Hkv, M, G;
    int num_pages, page_size, max_pages, max_len;
    int causal, window;
    float scale_log2;  // logit scale (and Q, K dequantization factors) times log2(e)
    float out_scale;   // V dequantization factor (1 for 16-bit caches)
    int chunk, S;
};

// ---- element types ---------------------------------------------------------
template <typename TI>
struct InT;
template <>
struct InT<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    // 16 bytes (8 elements) to floats: a BF16 value is the top half of its float
    __device__ static void cvt16(const uint4& w, float* f) {
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            f[2 * u] = __uint_as_float(x[u] << 16);
            f[2 * u + 1] = __uint_as_float(x[u] & 0xFFFF0000u);
        }
    }
    __device__ static float one(const void* p, size_t idx) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[idx]);
    }
    __device__ static float round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
};
template <>
struct InT<__half> {
    static constexpr int kBytes = 2;
    __device__ static void cvt16(const uint4& w, float* f) {
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&x[u]));
            f[2 * u] = t.x;
            f[2 * u + 1] = t.y;
        }
    }
    __device__ static float one(const void* p, size_t idx) {
        return __half2float(reinterpret_cast<const __half*>(p)[idx]);
    }
    __device__ static float round(float x) { return __half2float(__float2half_rn(x)); }
};
template <>
struct InT<E4M3In> {
    static constexpr int kBytes = 1;
    __device__ static float2 pair(uint32_t two) {
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
        return __half22float2(*reinterpret_cast<const __half2*>(&h));
    }
    __device__ static void cvt16(const uint4& w, float* f) {
        const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 lo = pair(x[u]), hi = pair(x[u] >> 16);
            f[4 * u] = lo.x;
            f[4 * u + 1] = lo.y;
            f[4 * u + 2] = hi.x;
            f[4 * u + 3] = hi.y;
        }
    }
    __device__ static float one(const void* p, size_t idx) {
        const __half_raw h =
            __nv_cvt_fp8_to_halfraw(reinterpret_cast<const __nv_fp8_storage_t*>(p)[idx], __NV_E4M3);
        return __half2float(__half(h));
    }
    // round to nearest E4M3 (saturating to the finite range), as the value product's operand
    __device__ static float round(float x) {
        const __nv_fp8_storage_t b = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
        return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
    }
};

template <typename TO>
__device__ __forceinline__ void store_out(void* o, size_t idx, float x);
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(void* o, size_t idx, float x) {
    reinterpret_cast<__nv_bfloat16*>(o)[idx] = __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ void store_out<__half>(void* o, size_t idx, float x) {
    reinterpret_cast<__half*>(o)[idx] = __float2half_rn(x);
}

__device__ __forceinline__ float gwarp_max(float x) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, s));
    return x;
}
__device__ __forceinline__ float gwarp_sum(float x) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    return x;
}

template <typename TI, typename TO, int D>
__global__ void __launch_bounds__(kGWarps * 32) attn_paged_group_kernel(const GroupArgs a) {
    using In = InT<TI>;
    constexpr int EPL = (D + 31) / 32;         // output elements per lane
    constexpr int VEC = 16 / In::kBytes;       // elements per 16-byte load
    constexpr int VPK = D / VEC;               // 16-byte loads per key row
    static_assert(D % VEC == 0, "a key row is a whole number of 16-byte loads");
    __shared__ float qs[kGWarps][D];
    __shared__ float ks[kGKeys][D + 1];  // +1: lane-per-key reads hit distinct banks
    __shared__ float vs[kGKeys][D];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int R = a.G * a.M;
    const int r = blockIdx.z * kGWarps + warp;
    const bool row_ok = r < R;
    const int h = g * a.G + (row_ok ? r / a.M : 0), i = row_ok ? r % a.M : 0;

    // this sequence's keys: L = clamp(seq_lens[b], 0, max_len); row i sits at
    // position i + L - M; the union of its rows' ranges is cut into splits
    // starting at the range's start rounded down to a 128-key tile
    const int L = min(max(__ldg(a.lens + b), 0), a.max_len);
    int lo0, hi0, lo1, hi1;
    key_range(L - a.M, L, a.causal, a.window, &lo0, &hi0);
    key_range(L - 1, L, a.causal, a.window, &lo1, &hi1);
    const int khi = max(hi1, lo0);
    const int kbase = (lo0 / kGTile) * kGTile;
    const int s_lo = kbase + split * a.chunk;
    const int s_hi = min(s_lo + a.chunk, khi);
    const int lo = max(lo0, s_lo);
    int r_lo = 0, r_hi = 0;  // this row's own visible keys
    if (row_ok) key_range(i + L - a.M, L, a.causal, a.window, &r_lo, &r_hi);

    const size_t qrow = ((size_t)b * a.Hq + h) * a.M + i;
    for (int d = lane; d < D; d += 32) qs[warp][d] = row_ok ? In::one(a.q, qrow * D + d) : 0.f;

    const int* trow = a.table + (size_t)b * a.max_pages;
    const uint8_t* kbytes = reinterpret_cast<const uint8_t*>(a.kp);
    const uint8_t* vbytes = reinterpret_cast<const uint8_t*>(a.vp);

    float m = -INFINITY, l = 0.f;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;

    for (int j0 = lo; j0 < s_hi; j0 += kGKeys) {
        __syncthreads();  // the previous tile consumed (and qs written)
        for (int x = threadIdx.x; x < kGKeys * VPK; x += kGWarps * 32) {
            const int kk = x / VPK, c = x % VPK;
            const int j = j0 + kk;
            uint4 wk = make_uint4(0u, 0u, 0u, 0u), wv = wk;  // all-zero bits are 0 in every input type
            if (j < s_hi) {
                const int page = __ldg(trow + j / a.page_size);
                // a table entry outside the pool reads as a page of zeros
                if (page >= 0 && page < a.num_pages) {
                    const size_t el = (((size_t)page * a.Hkv + g) * a.page_size + j % a.page_size) * D + c * VEC;
                    wk = __ldg(reinterpret_cast<const uint4*>(kbytes + el * In::kBytes));
                    wv = __ldg(reinterpret_cast<const uint4*>(vbytes + el * In::kBytes));
                }
            }
            float f[VEC];
            In::cvt16(wk, f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) ks[kk][c * VEC + e] = f[e];
            In::cvt16(wv, f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) vs[kk][c * VEC + e] = f[e];
        }
        __syncthreads();
        if (row_ok) {
            const int j = j0 + lane;
            float t = -INFINITY;  // masked and padded keys score -inf
            if (j < s_hi && j >= r_lo && j < r_hi) {
                float dot = 0.f;
#pragma unroll 8
                for (int d = 0; d < D; ++d) dot = fmaf(qs[warp][d], ks[lane][d], dot);
                t = dot * a.scale_log2;
            }
            const float m_new = fmaxf(m, gwarp_max(t));
            // ghost-row pin: while every key so far is masked, 0 stands for the maximum
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = exp2f(m - m_use);
            const float p = exp2f(t - m_use);
            l = l * alpha + gwarp_sum(p);
            // the value product takes P rounded to the input type; the row sum does not
            const float pr = In::round(p);
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
#pragma unroll 4
            for (int jj = 0; jj < kGKeys; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, pr, jj);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const int d = lane + 32 * e;
                    if (d < D) acc[e] = fmaf(pj, vs[jj][d], acc[e]);
                }
            }
            m = m_new;
        }
    }

    if (!row_ok) return;
    if (a.S > 1) {
        const size_t slot = qrow * a.S + split;
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
        const float inv = l > 0.f ? a.out_scale / l : 0.f;  // no visible key: output 0
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int d = lane + 32 * e;
            if (d < D) store_out<TO>(a.o, qrow * D + d, acc[e] * inv);
        }
    }
}

template <typename TI, typename TO>
cudaError_t launch_group_d(const GroupArgs& a, int D, dim3 grid, cudaStream_t stream) {
    switch (D) {
        case 16: attn_paged_group_kernel<TI, TO, 16><<<grid, kGWarps * 32, 0, stream>>>(a); break;
        case 32: attn_paged_group_kernel<TI, TO, 32><<<grid, kGWarps * 32, 0, stream>>>(a); break;
        case 64: attn_paged_group_kernel<TI, TO, 64><<<grid, kGWarps * 32, 0, stream>>>(a); break;
        case 128: attn_paged_group_kernel<TI, TO, 128><<<grid, kGWarps * 32, 0, stream>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

bool paged_tc_supported(const Problem& p, bool e4m3) { return decode_tc_supported(p) && (!e4m3 || p.D == 128); }

bool paged_group_supported(const Problem& p) {
    return (p.D == 16 || p.D == 32 || p.D == 64 || p.D == 128) &&
           ((long long)p.G * p.M + kGWarps - 1) / kGWarps <= 65535;
}

// Splits of whole 128-key tiles over the longest range any sequence can have
// (the plan must hold for every length up to kv.max_len), enough of them that
// the grid holds about four blocks per SM.
int paged_group_plan(const Problem& p, const PagedKV& kv, int* chunk, int* S) {
    long long tiles = ((long long)kv.max_len + kGTile - 1) / kGTile;
    if (p.window > 0) {
        const long long span = (long long)p.window + p.M - 1 + (kGTile - 1);
        const long long wt = (span + kGTile - 1) / kGTile;
        if (wt < tiles) tiles = wt;
    }
    if (tiles < 1) tiles = 1;
    const long long z = ((long long)p.G * p.M + kGWarps - 1) / kGWarps;
    const long long groups = (long long)p.B * p.Hkv * z;
    int sms = device_sm_count();
    if (sms <= 0) sms = 148;
    const long long target = 4LL * sms;
    long long s = groups > 0 ? (target + groups - 1) / groups : 1;
    if (s < 1) s = 1;
    if (s > tiles) s = tiles;
    if (s > 1024) s = 1024;
    const long long c = (tiles + s - 1) / s;
    *chunk = (int)(c * kGTile);
    *S = (int)((tiles + c - 1) / c);
    return ATTN_OK;
}

cudaError_t launch_paged_group(const Problem& p, const void* q, const PagedKV& kv, int chunk, int S,
                               const SplitWorkspace* ws, void* o, float out_scale, bool e4m3,
                               cudaStream_t stream) {
    GroupArgs a;
    a.q = q;
    a.kp = kv.k_pages;
    a.vp = kv.v_pages;
    a.table = kv.block_table;
    a.lens = kv.seq_lens;
    a.o = o;
    a.ws_m = ws ? ws->m : nullptr;
    a.ws_l = ws ? ws->l : nullptr;
    a.ws_acc = ws ? ws->acc : nullptr;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.M = p.M;
    a.G = p.G;
    a.num_pages = kv.num_pages;
    a.page_size = kv.page_size;
    a.max_pages = kv.max_pages;
    a.max_len = kv.max_len;
    a.causal = p.causal;
    a.window = p.window;
    a.scale_log2 = p.scale_log2;
    a.out_scale = out_scale;
    a.chunk = chunk;
    a.S = S;
    if (S > 1 && !ws) return cudaErrorInvalidValue;
    const int z = (p.G * p.M + kGWarps - 1) / kGWarps;
    const dim3 grid((unsigned)S, (unsigned)(p.B * p.Hkv), (unsigned)z);
    if (e4m3)
        return p.dtype == ATTN_BF16 ? launch_group_d<E4M3In, __nv_bfloat16>(a, p.D, grid, stream)
                                    : launch_group_d<E4M3In, __half>(a, p.D, grid, stream);
    return p.dtype == ATTN_BF16 ? launch_group_d<__nv_bfloat16, __nv_bfloat16>(a, p.D, grid, stream)
                                : launch_group_d<__half, __half>(a, p.D, grid, stream);
}

}  // namespace attn
