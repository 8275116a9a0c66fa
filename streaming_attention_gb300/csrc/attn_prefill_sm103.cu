// Prefill forward on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// One CTA owns two 128-row query tiles of one (batch, head) and streams the
// key/value tiles they may see. Warp roles:
//   warps 0-3  softmax for query tile 0 (one TMEM lane = one row = one thread)
//   warps 4-7  softmax for query tile 1
//   warp 8     TMA producer: Q once, then K_j, V_j through a shared-memory ring
//   warp 9     MMA issuer (one thread): S_t = Q_t K_j^T and O_t += P_t V_j
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [384,384+D).
// P_t (16-bit, two per column) overwrites the first 64 columns of S_t.
//
// The two query tiles ping-pong: while the softmax warps of one tile work on
// its score tile, the tensor core multiplies the other tile's scores, so the
// exponentials overlap the MMAs. Each row carries its running (m, l) in
// registers and its accumulator in TMEM, and never holds more than one
// 128-key tile of scores ("Compare reasoning after your own attempt",
// central-idea table, A3 row). Masked and padded keys score -inf ("Kernel
// Notes & Checklist", gotchas ledger), a row whose keys are all masked so far
// uses 0 as its maximum so it never forms -inf - (-inf) (same ledger, ghost
// rows), and only tiles that cross a mask edge pay for masking (same ledger,
// boundary checks are not free). Key tiles that no row of the CTA may see are
// never loaded (causal and window tile skipping).
//
// Rescaling is lazy: a row's reference maximum moves only when the new
// maximum exceeds it by more than 8 (base-2 units), so p = 2^(t - m_ref) <= 256
// and the accumulator is rescaled by alpha = 2^(m_old - m_new) only then. The
// final O / l is the same quotient as with an always-current maximum.
//
// Every wait is bounded (1 s); on expiry the CTA raises an abort flag, sets
// the device status word, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#include <mutex>

#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "tma_map.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;  // rows per query tile
constexpr int BN = 128;  // keys per key/value tile
constexpr int NQ = 2;    // query tiles per CTA
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;            // 128-byte swizzle chunks along D
    static constexpr int kChunkBytes = BM * 128;      // one chunk of a 128-row tile
    static constexpr int kTileBytes = BM * D * 2;     // one Q, K or V tile
    static constexpr int kStages = (D == 128) ? 4 : 8;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = NQ * kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
};

// TMEM column of S_t / P_t and of O_t
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }

struct PrefillParams {
    void* o;
    int* status;
    int M, N, Hq, Hkv, G;
    int causal, window;
    float scale_log2;
};

struct Shared {
    uint32_t bar_q, bar_full0, bar_empty0, bar_s0, bar_p0, bar_o;
    __device__ uint32_t full(int s) const { return bar_full0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar_empty0 + 8u * s; }
    __device__ uint32_t s_full(int t) const { return bar_s0 + 8u * t; }
    __device__ uint32_t p_full(int t) const { return bar_p0 + 8u * t; }
};

// Single-thread bounded wait. abortable: give up as soon as another thread raised the abort flag.
__device__ bool wait_one(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status,
                         bool abortable = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abortable && *abort_flag) return false;
        if (globaltimer_ns() - t0 > kTimeoutNs) {
            *abort_flag = 1u;
            atomicExch(status, 1);
            return false;
        }
    }
}

// Warp-uniform bounded wait: every lane observes the phase, and the whole
// warp gives up together.
__device__ bool wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        int stop = 0;
        if (lane == 0) {
            if (*abort_flag) {
                stop = 1;
            } else if (globaltimer_ns() - t0 > kTimeoutNs) {
                *abort_flag = 1u;
                atomicExch(status, 1);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kBF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kQOff;
    const uint32_t sKV = sbase + C::kKVOff;
    Shared sh;
    sh.bar_q = sbase + C::kBarOff;
    sh.bar_full0 = sh.bar_q + 8;
    sh.bar_empty0 = sh.bar_full0 + 8 * C::kStages;
    sh.bar_s0 = sh.bar_empty0 + 8 * C::kStages;
    sh.bar_p0 = sh.bar_s0 + 16;
    sh.bar_o = sh.bar_p0 + 16;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- which rows and keys this CTA owns --------------------------------
    const int bh = blockIdx.x;
    const int qb = gridDim.y - 1 - blockIdx.y;  // longest (causal) blocks first
    const int b = bh / p.Hq, h = bh % p.Hq;
    const int kvh = b * p.Hkv + h / p.G;
    const int row0 = qb * (NQ * BM);
    const int off = p.N - p.M;  // row i sits at key position i + off
    const int last_row = min(row0 + NQ * BM - 1, p.M - 1);
    int klo = 0, khi = p.N, lo_unused = 0, hi_unused = 0;
    key_range(row0 + off, p.N, p.causal, p.window, &klo, &hi_unused);
    key_range(last_row + off, p.N, p.causal, p.window, &lo_unused, &khi);
    const int jt0 = klo / BN;
    const int n = (khi > klo) ? (khi + BN - 1) / BN - jt0 : 0;  // key tiles to visit

    if (threadIdx.x == 0) {
        mbar_init(sh.bar_q, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(sh.full(s), 1);
            mbar_init(sh.empty(s), 1);
        }
        for (int t = 0; t < NQ; ++t) {
            mbar_init(sh.s_full(t), 1);
            mbar_init(sh.p_full(t), 4 * 32);
        }
        mbar_init(sh.bar_o, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kLoadWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(sh.bar_q, NQ * C::kTileBytes);
            for (int t = 0; t < NQ; ++t)
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tmQ, c * 64, row0 + t * BM, bh,
                                sh.bar_q);
            int issued = 0;
            // K_j and V_j alternate through the ring in the order the MMA uses them
            for (int u = 0; u < 2 * n; ++u) {
                const int s = u % C::kStages;
                if (u >= C::kStages &&
                    !wait_one(sh.empty(s), ((u / C::kStages) - 1) & 1, abort_flag, p.status))
                    break;
                mbar_arrive_expect_tx(sh.full(s), C::kTileBytes);
                const CUtensorMap* tm = (u & 1) ? &tmV : &tmK;
                const int key0 = (jt0 + u / 2) * BN;
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sKV + s * C::kTileBytes + c * C::kChunkBytes, tm, c * 64, key0, kvh, sh.full(s));
                issued = u + 1;
            }
            // every issued copy must land before the CTA may exit
            wait_one(sh.bar_q, 0, abort_flag, p.status, false);
            for (int u = max(0, issued - C::kStages); u < issued; ++u)
                wait_one(sh.full(u % C::kStages), (u / C::kStages) & 1, abort_flag, p.status, false);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0 && n > 0) {
            constexpr uint32_t idS = idesc_f16(kBF16, BM, BN, false);
            constexpr uint32_t idPV = idesc_f16(kBF16, BM, D, true);
            auto issue_s = [&](int t, int slot) {
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off_k = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
                    const uint64_t a = sw128_desc(sQ + t * C::kTileBytes + off_k, 16, 1024);
                    const uint64_t bd = sw128_desc(sKV + slot * C::kTileBytes + off_k, 16, 1024);
                    mma_ss(tmem + col_s(t), a, bd, idS, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int slot, bool first) {
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint64_t bd = sw128_desc(sKV + slot * C::kTileBytes + kk * 16 * 128, C::kChunkBytes, 1024);
                    mma_ts(tmem + col_o(t), tmem + col_s(t) + kk * 8, bd, idPV, (first && kk == 0) ? 0u : 1u);
                }
            };
            bool ok = wait_one(sh.bar_q, 0, abort_flag, p.status);
            tc_fence_after();
            int slot_v_prev = 0;
            for (int jj = 0; ok && jj < n; ++jj) {
                const int uk = 2 * jj, sk = uk % C::kStages;
                if (!(ok = wait_one(sh.full(sk), (uk / C::kStages) & 1, abort_flag, p.status))) break;
                tc_fence_after();
                issue_s(0, sk);
                mma_commit(sh.s_full(0));
                if (jj > 0) {
                    if (!(ok = wait_one(sh.p_full(1), (jj - 1) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    issue_pv(1, slot_v_prev, jj - 1 == 0);
                    mma_commit(sh.empty(slot_v_prev));
                }
                issue_s(1, sk);
                mma_commit(sh.s_full(1));
                mma_commit(sh.empty(sk));
                const int uv = 2 * jj + 1, sv = uv % C::kStages;
                if (!(ok = wait_one(sh.full(sv), (uv / C::kStages) & 1, abort_flag, p.status))) break;
                if (!(ok = wait_one(sh.p_full(0), jj & 1, abort_flag, p.status))) break;
                tc_fence_after();
                issue_pv(0, sv, jj == 0);
                slot_v_prev = sv;
            }
            if (ok && wait_one(sh.p_full(1), (n - 1) & 1, abort_flag, p.status)) {
                tc_fence_after();
                issue_pv(1, slot_v_prev, n - 1 == 0);
                mma_commit(sh.empty(slot_v_prev));
            }
            // all MMAs done -> O final (and TMEM/smem safe to release)
            mma_commit(sh.bar_o);
            wait_one(sh.bar_o, 0, abort_flag, p.status, false);
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps ----------------
        const int t = warp >> 2;            // query tile
        const int wq = warp & 3;            // TMEM lane quarter
        const int r_in_tile = wq * 32 + lane;
        const int row = row0 + t * BM + r_in_tile;
        const int pos = row + off;
        const int tile_first_pos = row0 + t * BM + off;
        const int tile_last_pos = tile_first_pos + BM - 1;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + col_s(t);
        const uint32_t tO = tmem + lane_base + col_o(t);
        const float c = p.scale_log2;
        const float masked_s = c >= 0.f ? -INFINITY : INFINITY;  // scores that give t = -inf

        float m_ref = -INFINITY;  // reference maximum (base-2 scaled units)
        float l = 0.f;
        bool ok = true;
        for (int jj = 0; jj < n; ++jj) {
            const int key0 = (jt0 + jj) * BN;
            if (!(ok = wait_warp(sh.s_full(t), jj & 1, abort_flag, p.status))) break;
            tc_fence_after();
            uint32_t s[4][32];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld_x32(tS + q4 * 32, s[q4]);
            tmem_wait_ld_x32(s[0]);
            reg_after_x32(s[1]);
            reg_after_x32(s[2]);
            reg_after_x32(s[3]);

            // mask only tiles that cross an edge (ragged N, causal diagonal, window start)
            const bool need_mask = (key0 + BN > p.N) || (p.causal && key0 + BN - 1 > tile_first_pos) ||
                                   (p.window > 0 && key0 <= tile_last_pos - p.window);
            if (need_mask) {
                int lo = 0, hi = 0;
                key_range(pos, p.N, p.causal, p.window, &lo, &hi);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int key = key0 + q4 * 32 + e;
                        if (key < lo || key >= hi) s[q4][e] = __float_as_uint(masked_s);
                    }
            }
            float mx;
            if (c >= 0.f) {
                mx = -INFINITY;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(s[q4][e]));
            } else {
                mx = INFINITY;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx = fminf(mx, __uint_as_float(s[q4][e]));
            }
            const float m_tile = mx * c;  // -inf when the whole tile is masked for this row
            const float m_new = fmaxf(m_ref, m_tile);
            const bool need = m_new > m_ref + kRescaleThreshold;
            float alpha = 1.f;
            if (need) {
                alpha = ex2(m_ref - m_new);  // m_ref = -inf -> 0
                l *= alpha;
                m_ref = m_new;
            }
            // ghost-row pin: while every key so far is masked, exponentiate against 0
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
            const float neg_m = -m_use;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t packed[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2(fmaf(__uint_as_float(s[q4][2 * e]), c, neg_m));
                    const float p1 = ex2(fmaf(__uint_as_float(s[q4][2 * e + 1]), c, neg_m));
                    l += p0 + p1;
                    packed[e] = pack2<kBF16>(p0, p1);
                }
                tmem_st_x16(tS + q4 * 16, packed);  // P overwrites the first 64 columns of S
            }
            // rescale the accumulator (the PV of the previous tile has completed:
            // its commit preceded this tile's score commit)
            if (__any_sync(0xffffffffu, need) && jj > 0) {
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld_x32(tO + ch * 32, o);
                    tmem_wait_ld_x32(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_x32(tO + ch * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(sh.p_full(t));
        }

        // ---------------- epilogue: O / l, one cast, store rows < M ----------------
        int stop = 0;
        if (lane == 0) stop = *abort_flag ? 1 : 0;
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (ok && !stop) {
            const bool have = n > 0 && wait_warp(sh.bar_o, 0, abort_flag, p.status);
            if (n == 0 || have) {
                tc_fence_after();
                const float inv = l > 0.f ? 1.f / l : 0.f;  // no visible key: output 0
                uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((size_t)bh * p.M + row) * D;
#pragma unroll
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    if (n > 0) {
                        tmem_ld_x32(tO + ch * 32, o);
                        tmem_wait_ld_x32(o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack2<kBF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    if (row < p.M) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4)
                            dst[v4] = make_uint4(w[4 * v4], w[4 * v4 + 1], w[4 * v4 + 2], w[4 * v4 + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
int launch_t(const Problem& pr, const void* q, const void* k, const void* v, void* o, int* status,
             cudaStream_t stream) {
    using C = Cfg<D>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_prefill_kernel<D, kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        C::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return ATTN_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (!make_tensor_map(&tq, q, D, pr.M, pr.B * pr.Hq, BM, kBF16) ||
        !make_tensor_map(&tk, k, D, pr.N, pr.B * pr.Hkv, BN, kBF16) ||
        !make_tensor_map(&tv, v, D, pr.N, pr.B * pr.Hkv, BN, kBF16))
        return ATTN_ERR_CUDA;
    PrefillParams pp;
    pp.o = o;
    pp.status = status;
    pp.M = pr.M;
    pp.N = pr.N;
    pp.Hq = pr.Hq;
    pp.Hkv = pr.Hkv;
    pp.G = pr.G;
    pp.causal = pr.causal;
    pp.window = pr.window;
    pp.scale_log2 = pr.scale_log2;
    dim3 grid(pr.B * pr.Hq, (pr.M + NQ * BM - 1) / (NQ * BM));
    attn_prefill_kernel<D, kBF16><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, pp);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

bool prefill_supported(const Problem& p) {
    return (p.D == 64 || p.D == 128) && (p.M + NQ * BM - 1) / (NQ * BM) <= 65535;
}

int launch_prefill(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                   cudaStream_t stream) {
    const bool bf16 = p.dtype == ATTN_BF16;
    if (p.D == 128) return bf16 ? launch_t<128, true>(p, q, k, v, o, status, stream)
                                : launch_t<128, false>(p, q, k, v, o, status, stream);
    if (p.D == 64) return bf16 ? launch_t<64, true>(p, q, k, v, o, status, stream)
                               : launch_t<64, false>(p, q, k, v, o, status, stream);
    return ATTN_ERR_HEADDIM;
}

}  // namespace attn
