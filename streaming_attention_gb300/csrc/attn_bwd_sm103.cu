// Backward pass of the streaming attention forward on the tcgen05 tensor
// cores (sm_103a), D in {64, 128}.
//
// With the forward's per-row log-sum-exp (lse) the weights of any (row, key)
// pair are recomputed exactly, P = exp(scale s - lse), so the backward needs
// no running state. Each row of dS is the softmax vector-Jacobian product of
// that row, dS = P * (dP - delta) with dP = dO V^T and delta = sum_j P dP =
// rowsum(dO * O) ("Intermediate and advanced kernel workshops", workshop I2,
// softmax backward; the answer key's I2 row: one FP32 reduction, then the
// probability-weighted difference). Then dV = P^T dO, dK = scale dS^T Q and
// dQ = scale dS K.
//
// Two kernels, each owning its outputs, so no output is ever accumulated
// across CTAs:
//   dK/dV kernel: one CTA per (128-key tile, KV head); K and V stay in shared
//     memory while the query tiles of all G query heads of the group stream
//     through a 2-stage TMA ring (Q, dO, and their rows' lse and delta).
//     S^T = K Q^T and dP^T = V dO^T land in TMEM (TMEM lane = key); the
//     elementwise warps turn them into P^T and dS^T (16-bit, written over the
//     first half of each), and the MMA warp accumulates dV += P^T dO and
//     dK += dS^T Q in TMEM. The elementwise warps keep their P^T in registers
//     for the dS^T pass, so the next tile's S^T may overwrite P^T as soon as
//     the dV product has read it.
//   dQ kernel: one CTA per (128-row query tile, query head); Q and dO stay,
//     K and V tiles stream; S = Q K^T and dP = dO V^T in TMEM (lane = row);
//     the elementwise warps take S into registers (which frees it for the next
//     tile's product at once) and keep P there; dS over dP, dQ += dS K.
// S and dP are thus computed twice (7 products instead of 5); in exchange
// neither kernel needs atomics or a transpose through shared memory. The dQ
// kernel reads nothing the dK/dV kernel writes, so it is launched
// programmatically: its CTAs start on the SMs the dK/dV grid's last wave
// leaves idle, and each waits for that grid only before it exits.
// The elementwise passes run on packed FP32 pairs (fma/add/mul.f32x2; the row
// statistics are stored negated for that), and each kernel's outputs leave
// through the idle stage ring as swizzled boxes stored by TMA.
// Tiles outside the causal / window range are skipped; only edge tiles mask.
// Every wait is bounded (1 s); on expiry a CTA sets the device status word,
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "tma_map.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BT = 128;           // query rows per query tile and keys per key tile
// warps 0-7 elementwise (warp w: TMEM lanes 32*(w%4).., column half w/4), 8 TMA, 9 MMA
constexpr int kBwdThreads = 320;
constexpr int kBLoadWarp = 8, kBMmaWarp = 9;
constexpr uint64_t kBwdTimeoutNs = 1000000000ull;

// Shared memory: two stationary tiles, a 2-stage ring of tile pairs, the
// per-row vectors of each stage (dK/dV kernel), barriers.
template <int D>
struct BCfg {
    static constexpr int kTile = BT * D * 2;  // one [128][D] 16-bit tile
    static constexpr int kChunk = BT * 128;   // one 64-column (128-byte) chunk of a tile
    static constexpr int kChunks = D / 64;
    static constexpr int kStages = 2;
    static constexpr int kOffStat = 0;                                  // 2 stationary tiles
    static constexpr int kOffStage = 2 * kTile;                         // stage s: 2 tiles at + s * 2 * kTile
    static constexpr int kOffVec = kOffStage + kStages * 2 * kTile;     // stage s: nlse2[128], ndelta[128]
    static constexpr int kOffBar = kOffVec + kStages * 2 * BT * 4;
    // stat_full, full[2], empty[2], st_full[2], p_full[2], done, drain, ep
    static constexpr int kNumBars = 1 + 2 * kStages + 7;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    // TMEM columns
    static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
};

struct BwdParams {
    void* out0;          // dK (dK/dV kernel) or dQ (dQ kernel)
    void* out1;          // dV (dK/dV kernel)
    // per-row statistics, negated so that the elementwise passes add them with packed
    // FMA/add instructions (which have no negated operand)
    const float* nlse2;   // [B*Hq][Mpad]: -lse * log2(e); +inf past M (those rows are masked)
    const float* ndelta;  // [B*Hq][Mpad]: -rowsum(dO * O); 0 past M
    int* status;
    int Hq, Hkv, M, N, G, Mpad;
    int causal, window;
    float scale, scale_log2;
    int groups;  // B * Hkv (dK/dV) or B * Hq (dQ)
    int ntile;   // key tiles (dK/dV) or query tiles (dQ)
};

__device__ bool bwait_one(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status,
                          bool abortable = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abortable && *abort_flag) return false;
        if (globaltimer_ns() - t0 > kBwdTimeoutNs) {
            *abort_flag = 1u;
            atomicExch(status, 1);
            return false;
        }
    }
}

__device__ bool bwait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        int stop = 0;
        if (lane == 0) {
            if (*abort_flag) {
                stop = 1;
            } else if (globaltimer_ns() - t0 > kBwdTimeoutNs) {
                *abort_flag = 1u;
                atomicExch(status, 1);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

// Warp-uniform bounded wait that ignores the abort flag (for the final drain).
__device__ bool bwait_warp_final(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        int stop = 0;
        if ((threadIdx.x & 31) == 0 && globaltimer_ns() - t0 > kBwdTimeoutNs) {
            atomicExch(status, 1);
            stop = 1;
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

// The MMA issuer is a whole warp: every lane runs the issuing loop, so operands
// stay warp-uniform, and one elected lane issues each MMA and commit (the _el
// forms). The two helpers below are called by that warp only.
// C = A B^T over D (both operands K-major [128][D] tiles, 128 x 128 result)
template <int D>
__device__ __forceinline__ void mma_rows_by_rows(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)((((kk >> 2) * BCfg<D>::kChunk) + (kk & 3) * 32) >> 4);
        mma_ss_el(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
    }
}
// A 16-bit operand of 128 along K lives in TMEM as two packed blocks: K 0..63 in
// columns [0, 32) and K 64..127 in columns [64, 96) of its region, each written
// in place over the 32-bit values of its own 64 columns by one elementwise
// warpgroup (so the two warpgroups never touch each other's columns).
__device__ __forceinline__ constexpr uint32_t packed_col(int q4) { return (q4 >> 1) * 64 + (q4 & 1) * 16; }

// C (+)= A B over 128: A 16-bit in TMEM (packed as above), B a [128][D] tile read
// MN-major (N = D)
__device__ __forceinline__ void mma_tmem_by_tile(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, uint32_t idesc,
                                                 bool first) {
#pragma unroll
    for (int kk = 0; kk < BT / 16; ++kk)
        mma_ts_el(d_tmem, a_tmem + (kk >> 2) * 64 + (kk & 3) * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4), idesc,
               (first && kk == 0) ? 0u : 1u);
}

// 16-bit pair (low half first) -> two floats
template <bool kBF16>
__device__ __forceinline__ void unpack2(uint32_t w, float& lo, float& hi) {
    if (kBF16) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xFFFF0000u);
    } else {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        lo = f.x;
        hi = f.y;
    }
}

template <bool kBF16>
__device__ __forceinline__ uint32_t bpack2(float lo, float hi) {
    return kBF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

// Output epilogue through shared memory: once the last product has completed,
// the stage ring is idle, so it holds the outputs as 128-row x 64-column boxes
// (16 KB each, in the TMA's 128-byte swizzle) that one thread stores with TMA
// copies (a row-per-thread global store touches 32 rows per instruction).
// Warp column half `half` owns columns [half D / 2, (half + 1) D / 2) of every
// output; this thread writes its lane's row r of them, times `mul`, as 16 bits.
template <int D, bool kBF16>
__device__ __forceinline__ void stage_row(uint32_t taddr, float mul, uint32_t boxes, int r, int half) {
    const uint64_t m2 = f2_pack(mul, mul);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        const int col0 = half * (D / 2) + c * 32;  // 32 columns per TMEM load
        uint32_t v[32];
        tmem_ld_x32(taddr + col0, v);
        tmem_wait_ld_x32(v);
        const uint32_t row = boxes + (col0 / 64) * (BT * 128) + r * 128;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {  // 16-byte chunk (col0 % 64) / 8 + c8 of the box row
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float y0, y1;
                f2_unpack(f2_mul(f2_pack(__uint_as_float(v[c8 * 8 + 2 * e]), __uint_as_float(v[c8 * 8 + 2 * e + 1])),
                                 m2),
                          y0, y1);
                w4[e] = kBF16 ? pack_bf16(y0, y1) : pack_f16(y0, y1);
            }
            const int chunk = (col0 % 64) / 8 + c8;
            st_shared_v4(row + ((chunk ^ (r & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
        }
    }
}

// Shared setup of both kernels: barriers, TMEM (512 columns), abort flag.
struct BSetup {
    uint32_t sbase, bar_stat, bar_full0, bar_empty0, bar_st0, bar_p0, bar_done, bar_drain, bar_ep, tmem;
    volatile uint32_t* abort_flag;
    __device__ uint32_t full(int s) const { return bar_full0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return bar_empty0 + 8u * s; }
    __device__ uint32_t st(int x) const { return bar_st0 + 8u * x; }  // x = 0: S computed; 1: dP computed
    // x = 0: P written (dK/dV kernel) or S taken into registers (dQ kernel); 1: dS written
    __device__ uint32_t pp(int x) const { return bar_p0 + 8u * x; }
};

template <int D>
__device__ __forceinline__ BSetup bwd_setup(uint8_t* smem) {
    using C = BCfg<D>;
    BSetup b;
    b.sbase = smem_u32(smem);
    b.bar_stat = b.sbase + C::kOffBar;
    b.bar_full0 = b.bar_stat + 8;
    b.bar_empty0 = b.bar_full0 + 8 * C::kStages;
    b.bar_st0 = b.bar_empty0 + 8 * C::kStages;
    b.bar_p0 = b.bar_st0 + 16;
    b.bar_done = b.bar_p0 + 16;
    b.bar_drain = b.bar_done + 8;
    b.bar_ep = b.bar_drain + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);
    b.abort_flag = tmem_slot + 1;
    if (threadIdx.x == 0) {
        mbar_init(b.bar_stat, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(b.full(s), 1);
            mbar_init(b.empty(s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(b.st(h), 1);
            mbar_init(b.pp(h), 8);  // one arrival per elementwise warp
        }
        mbar_init(b.bar_done, 1);
        mbar_init(b.bar_drain, 1);
        mbar_init(b.bar_ep, 8);  // one arrival per elementwise warp: its output rows are staged
        *b.abort_flag = 0u;
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == kBMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    b.tmem = *tmem_slot;
    return b;
}

__device__ __forceinline__ void bwd_teardown(const BSetup& b) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == kBMmaWarp) {
        tc_fence_after();
        tmem_dealloc(b.tmem, 512);
    }
}

// Thread 0 stores the staged boxes (per output, D / 64 boxes of 64 columns) once
// all eight elementwise warps have arrived, then waits for the copies to complete.
template <int D>
__device__ __forceinline__ void store_boxes(const BSetup& b, uint32_t boxes, const CUtensorMap* out0,
                                            const CUtensorMap* out1, int nout, int row0, int z, int* status) {
    if (threadIdx.x != 0) return;
    const bool ready = bwait_one(b.bar_ep, 0, b.abort_flag, status);
    if (!ready || *b.abort_flag) return;
    constexpr int per = D / 64;
    for (int o = 0; o < nout; ++o)
        for (int h = 0; h < per; ++h)
            tma_store_3d(o ? out1 : out0, boxes + (o * per + h) * (BT * 128), h * 64, row0, z);
    bulk_commit();
    bulk_wait_all();
}

// ---------------------------------------------------------------------------
// dK / dV: one CTA per (128-key tile, KV head)
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                         const BwdParams p) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // The dQ kernel (launched after this one, programmatically) reads nothing this
    // kernel writes: its CTAs may start on SMs this grid's last wave leaves idle.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const BSetup bs = bwd_setup<D>(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The key tiles of one group are consecutive CTAs, so the CTAs running at once
    // share a few groups' Q and dO in L2; each starts its walk over the query
    // tiles at a different tile, so at any moment they fetch different tiles (one
    // DRAM read each, then L2 hits) instead of all missing on the same one.
    const int jt = blockIdx.x % p.ntile, grp = blockIdx.x / p.ntile;
    const int b = grp / p.Hkv, g = grp % p.Hkv;
    const int k0 = jt * BT, k1 = min(k0 + BT, p.N);
    const int off = p.N - p.M;  // query row i sits at key position i + off
    // query rows that see a key of [k0, k1): causal needs i + off >= k0, a window
    // needs i + off < (k1 - 1) + window
    int i_lo = 0, i_hi = p.M;
    if (p.causal) i_lo = max(0, k0 - off);
    if (p.window > 0) i_hi = min(p.M, k1 - 1 + p.window - off);
    const int qt0 = i_lo / BT;
    const int nq = i_hi > i_lo ? (i_hi + BT - 1) / BT - qt0 : 0;
    const int T = p.G * nq;  // (query head of the group, query tile) pairs
    const int rot = T > 0 ? (int)(((long long)jt * 7) % T) : 0;

    if (warp == kBLoadWarp) {
        if (lane == 0 && T > 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmdO);
            mbar_arrive_expect_tx(bs.bar_stat, 2 * C::kTile);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(bs.sbase + C::kOffStat + c * C::kChunk, &tmK, c * 64, k0, grp, bs.bar_stat);
                tma_load_3d(bs.sbase + C::kOffStat + C::kTile + c * C::kChunk, &tmV, c * 64, k0, grp, bs.bar_stat);
            }
            int issued = 0;
            for (int it = 0; it < T; ++it) {
                const int s = it & 1;
                if (it >= 2 && !bwait_one(bs.empty(s), ((it >> 1) - 1) & 1, bs.abort_flag, p.status)) break;
                const int x = (it + rot) % T;
                const int h = g * p.G + x / nq, i0 = (qt0 + x % nq) * BT;
                const int bh = b * p.Hq + h;
                mbar_arrive_expect_tx(bs.full(s), 2 * C::kTile + 2 * BT * 4);
                const uint32_t dq = bs.sbase + C::kOffStage + s * 2 * C::kTile;
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(dq + c * C::kChunk, &tmQ, c * 64, i0, bh, bs.full(s));
                    tma_load_3d(dq + C::kTile + c * C::kChunk, &tmdO, c * 64, i0, bh, bs.full(s));
                }
                const uint32_t vec = bs.sbase + C::kOffVec + s * 2 * BT * 4;
                bulk_g2s(vec, p.nlse2 + (size_t)bh * p.Mpad + i0, BT * 4, bs.full(s));
                bulk_g2s(vec + BT * 4, p.ndelta + (size_t)bh * p.Mpad + i0, BT * 4, bs.full(s));
                issued = it + 1;
            }
            // every issued copy lands before the CTA may exit
            bwait_one(bs.bar_stat, 0, bs.abort_flag, p.status, false);
            for (int x = max(0, issued - 2); x < issued; ++x)
                bwait_one(bs.full(x & 1), (x >> 1) & 1, bs.abort_flag, p.status, false);
        }
    } else if (warp == kBMmaWarp) {
        if (T > 0) {  // the whole warp (see mma_rows_by_rows)
            constexpr uint32_t idS = idesc_f16(kBF16, BT, BT, false);
            constexpr uint32_t idAcc = idesc_f16(kBF16, BT, D, true);
            const uint64_t dK = sw128_desc(bs.sbase + C::kOffStat, 16, 1024);
            const uint64_t dV = sw128_desc(bs.sbase + C::kOffStat + C::kTile, 16, 1024);
            // Two-phase pipeline: S^T and dP^T of a tile are full 128-wide products; the
            // elementwise warps write P^T over S^T (phase A) while dP^T is computed, then
            // dS^T over dP^T (phase B), taking P^T from their registers. dV needs only
            // phase A, and the next tile's S^T follows dV at once, ahead of phase B and
            // of this tile's dK product.
            auto stage_q = [&](int it) { return bs.sbase + C::kOffStage + (it & 1) * 2 * C::kTile; };
            auto issue_s = [&](int it) {  // S^T = K Q^T
                mma_rows_by_rows<D>(bs.tmem + C::kColS, dK, sw128_desc(stage_q(it), 16, 1024), idS);
                mma_commit_el(bs.st(0));
            };
            auto issue_dp = [&](int it) {  // dP^T = V dO^T
                mma_rows_by_rows<D>(bs.tmem + C::kColDP, dV, sw128_desc(stage_q(it) + C::kTile, 16, 1024), idS);
                mma_commit_el(bs.st(1));
            };
            bool ok = bwait_warp(bs.bar_stat, 0, bs.abort_flag, p.status) &&
                      bwait_warp(bs.full(0), 0, bs.abort_flag, p.status);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
            }
            for (int it = 0; ok && it < T; ++it) {
                const uint32_t sq = stage_q(it);
                if (!(ok = bwait_warp(bs.pp(0), it & 1, bs.abort_flag, p.status))) break;
                tc_fence_after();
                mma_tmem_by_tile(bs.tmem + C::kColAcc1, bs.tmem + C::kColS, sw128_desc(sq + C::kTile, C::kChunk, 1024),
                                 idAcc, it == 0);  // dV += P^T dO
                // the next S^T may overwrite P^T now: dV reads it first (same pipe), and
                // phase B takes P from the elementwise warps' registers
                const bool more = it + 1 < T;
                if (more) {
                    if (!(ok = bwait_warp(bs.full((it + 1) & 1), ((it + 1) >> 1) & 1, bs.abort_flag, p.status))) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
                if (!(ok = bwait_warp(bs.pp(1), it & 1, bs.abort_flag, p.status))) break;
                tc_fence_after();
                mma_tmem_by_tile(bs.tmem + C::kColAcc0, bs.tmem + C::kColDP, sw128_desc(sq, C::kChunk, 1024), idAcc,
                                 it == 0);  // dK += dS^T Q
                mma_commit_el(bs.empty(it & 1));  // Q, dO of this tile fully read
                if (more) issue_dp(it + 1);
            }
            if (ok) mma_commit_el(bs.bar_done);
            mma_commit_el(bs.bar_drain);
            bwait_warp_final(bs.bar_drain, 0, p.status);
        }
        __syncwarp();
    } else {
        // elementwise: thread = key of the tile (TMEM lane); columns = query rows
        const int kl = (warp & 3) * 32 + lane, half = warp >> 2;  // key; column half of the tile
        const int key = k0 + kl;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const float c = p.scale_log2;
        bool ok = true;
        for (int it = 0; ok && it < T; ++it) {
            const int s = it & 1;
            const int i0 = (qt0 + (it + rot) % T % nq) * BT;
            uint32_t pkeep[2][16];  // this thread's packed P of phase A, used again by phase B
            const bool need_mask = (i0 + BT > p.M) || (k0 + BT > p.N) ||
                                   (p.causal && k0 + BT - 1 > i0 + off) ||
                                   (p.window > 0 && k0 <= i0 + BT - 1 + off - p.window);
            const float* nlse2 = reinterpret_cast<const float*>(smem + C::kOffVec + s * 2 * BT * 4);
            const float* ndel = nlse2 + BT;
            const uint64_t c2 = f2_pack(c, c);
            // ---- phase A: P^T = exp2(S^T c - lse2), packed over S^T ----
            if (!(ok = bwait_warp(bs.st(0), it & 1, bs.abort_flag, p.status))) break;
            // the stage's row vectors came by bulk copy: observe their barrier too (its
            // phase cannot move on before this tile's products, which need this thread)
            if (!(ok = bwait_warp(bs.full(s), (it >> 1) & 1, bs.abort_flag, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int q4 = 2 * half + qq, c0 = q4 * 32;  // TMEM column = query row of the tile
                uint32_t sv[32];
                tmem_ld_x32(bs.tmem + lane_base + C::kColS + c0, sv);
                tmem_wait_ld_x32(sv);
                // visible query rows of this chunk for this thread's key: e in [elo, ehi)
                int elo = 0, ehi = 32;
                if (need_mask) {
                    const int r0 = i0 + c0;  // row of e = 0, at position r0 + off
                    if (key >= p.N) ehi = 0;
                    ehi = min(ehi, p.M - r0);
                    if (p.causal) elo = max(elo, key - r0 - off);
                    if (p.window > 0) ehi = min(ehi, key + p.window - r0 - off);
                }
                uint32_t pk[16];
                auto chunk = [&](auto masked) {
#pragma unroll
                    for (int g4 = 0; g4 < 8; ++g4) {
                        const float4 l4 = reinterpret_cast<const float4*>(nlse2 + c0)[g4];
                        const int e = g4 * 4;
                        float x[4], pr[4];
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2,
                                         f2_pack(l4.x, l4.y)),
                                  x[0], x[1]);
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), c2,
                                         f2_pack(l4.z, l4.w)),
                                  x[2], x[3]);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            float pv = ex2(x[u]);
                            if (decltype(masked)::value) pv = (e + u >= elo && e + u < ehi) ? pv : 0.f;
                            pr[u] = pv;
                        }
                        pk[2 * g4] = bpack2<kBF16>(pr[0], pr[1]);
                        pk[2 * g4 + 1] = bpack2<kBF16>(pr[2], pr[3]);
                    }
                };
                if (need_mask)
                    chunk(std::true_type{});
                else
                    chunk(std::false_type{});
                tmem_st_x16(bs.tmem + lane_base + C::kColS + packed_col(q4), pk);
#pragma unroll
                for (int x = 0; x < 16; ++x) pkeep[qq][x] = pk[x];
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();  // the warp's TMEM stores before lane 0's arrival
            if ((threadIdx.x & 31) == 0) mbar_arrive(bs.pp(0));
            // ---- phase B: dS^T = P^T (dP^T - delta), packed over dP^T ----
            // (masked entries have P = 0 already)
            if (!(ok = bwait_warp(bs.st(1), it & 1, bs.abort_flag, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int q4 = 2 * half + qq, c0 = q4 * 32;
                uint32_t dpv[32];
                tmem_ld_x32(bs.tmem + lane_base + C::kColDP + c0, dpv);
                tmem_wait_ld_x32(dpv);
                const uint32_t* pv16 = pkeep[qq];
                uint32_t dk[16];
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const float4 d4 = reinterpret_cast<const float4*>(ndel + c0)[g4];
                    float p0, p1, p2, p3, y0, y1, y2, y3;
                    unpack2<kBF16>(pv16[2 * g4], p0, p1);
                    unpack2<kBF16>(pv16[2 * g4 + 1], p2, p3);
                    const int e = g4 * 4;
                    f2_unpack(f2_mul(f2_pack(p0, p1), f2_add(f2_pack(__uint_as_float(dpv[e]), __uint_as_float(dpv[e + 1])),
                                                             f2_pack(d4.x, d4.y))),
                              y0, y1);
                    f2_unpack(f2_mul(f2_pack(p2, p3),
                                     f2_add(f2_pack(__uint_as_float(dpv[e + 2]), __uint_as_float(dpv[e + 3])),
                                            f2_pack(d4.z, d4.w))),
                              y2, y3);
                    dk[2 * g4] = bpack2<kBF16>(y0, y1);
                    dk[2 * g4 + 1] = bpack2<kBF16>(y2, y3);
                }
                tmem_st_x16(bs.tmem + lane_base + C::kColDP + packed_col(q4), dk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();  // the warp's TMEM stores before lane 0's arrival
            if ((threadIdx.x & 31) == 0) mbar_arrive(bs.pp(1));
        }
        uint16_t* dk_row = reinterpret_cast<uint16_t*>(p.out0) + ((size_t)grp * p.N + key) * D;
        uint16_t* dv_row = reinterpret_cast<uint16_t*>(p.out1) + ((size_t)grp * p.N + key) * D;
        const bool write = key < p.N;
        if (T == 0) {  // no query row sees these keys: zero gradients
            if (write) {
#pragma unroll
                for (int x = half * (D / 16); x < (half + 1) * (D / 16); ++x) {
                    reinterpret_cast<uint4*>(dk_row)[x] = make_uint4(0, 0, 0, 0);
                    reinterpret_cast<uint4*>(dv_row)[x] = make_uint4(0, 0, 0, 0);
                }
            }
        } else {
            const uint32_t boxes = bs.sbase + C::kOffStage;  // dK boxes, then dV boxes
            if (ok && bwait_warp(bs.bar_done, 0, bs.abort_flag, p.status)) {
                tc_fence_after();
                stage_row<D, kBF16>(bs.tmem + lane_base + C::kColAcc0, p.scale, boxes, kl, half);
                stage_row<D, kBF16>(bs.tmem + lane_base + C::kColAcc1, 1.f, boxes + (D / 64) * BT * 128, kl, half);
                fence_proxy_async_smem();  // the boxes are read by the TMA (async proxy)
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bs.bar_ep);  // every warp arrives, also after giving up
            store_boxes<D>(bs, boxes, &tmdK, &tmdV, 2, k0, grp, p.status);
        }
    }
    bwd_teardown(bs);
}

// ---------------------------------------------------------------------------
// dQ: one CTA per (128-row query tile, query head)
// ---------------------------------------------------------------------------
template <int D, bool kBF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmdQ, const BwdParams p) {
    using C = BCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BSetup bs = bwd_setup<D>(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The query tiles of one head are consecutive CTAs (the last, under a causal
    // mask the longest, first) so the CTAs running at once share its K and V in
    // L2; each starts its walk over the key tiles at a different tile.
    const int qt = p.ntile - 1 - (int)(blockIdx.x % p.ntile), bh = blockIdx.x / p.ntile;
    const int b = bh / p.Hq, h = bh % p.Hq;
    const int grp = b * p.Hkv + h / p.G;
    const int i0 = qt * BT, i_last = min(i0 + BT, p.M) - 1;
    const int off = p.N - p.M;
    int lo = 0, hi = 0, unused = 0;
    key_range(i0 + off, p.N, p.causal, p.window, &lo, &unused);
    key_range(i_last + off, p.N, p.causal, p.window, &unused, &hi);
    const int kt0 = lo / BT;
    const int T = hi > lo ? (hi + BT - 1) / BT - kt0 : 0;  // key tiles
    const int rot = T > 0 ? (int)(((long long)qt * 7) % T) : 0;

    if (warp == kBLoadWarp) {
        if (lane == 0 && T > 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmdO);
            mbar_arrive_expect_tx(bs.bar_stat, 2 * C::kTile);
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_3d(bs.sbase + C::kOffStat + c * C::kChunk, &tmQ, c * 64, i0, bh, bs.bar_stat);
                tma_load_3d(bs.sbase + C::kOffStat + C::kTile + c * C::kChunk, &tmdO, c * 64, i0, bh, bs.bar_stat);
            }
            int issued = 0;
            for (int it = 0; it < T; ++it) {
                const int s = it & 1;
                if (it >= 2 && !bwait_one(bs.empty(s), ((it >> 1) - 1) & 1, bs.abort_flag, p.status)) break;
                const int k0 = (kt0 + (it + rot) % T) * BT;
                mbar_arrive_expect_tx(bs.full(s), 2 * C::kTile);
                const uint32_t dk = bs.sbase + C::kOffStage + s * 2 * C::kTile;
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_3d(dk + c * C::kChunk, &tmK, c * 64, k0, grp, bs.full(s));
                    tma_load_3d(dk + C::kTile + c * C::kChunk, &tmV, c * 64, k0, grp, bs.full(s));
                }
                issued = it + 1;
            }
            bwait_one(bs.bar_stat, 0, bs.abort_flag, p.status, false);
            for (int x = max(0, issued - 2); x < issued; ++x)
                bwait_one(bs.full(x & 1), (x >> 1) & 1, bs.abort_flag, p.status, false);
        }
    } else if (warp == kBMmaWarp) {
        if (T > 0) {  // the whole warp (see mma_rows_by_rows)
            constexpr uint32_t idS = idesc_f16(kBF16, BT, BT, false);
            constexpr uint32_t idAcc = idesc_f16(kBF16, BT, D, true);
            const uint64_t dQ = sw128_desc(bs.sbase + C::kOffStat, 16, 1024);
            const uint64_t ddO = sw128_desc(bs.sbase + C::kOffStat + C::kTile, 16, 1024);
            // Two-phase pipeline: full 128-wide S and dP; phase A takes S into registers,
            // which frees S for the next tile's product at once, and keeps P there; phase B
            // writes dS over dP.
            auto stage_k = [&](int it) { return bs.sbase + C::kOffStage + (it & 1) * 2 * C::kTile; };
            auto issue_s = [&](int it) {  // S = Q K^T
                mma_rows_by_rows<D>(bs.tmem + C::kColS, dQ, sw128_desc(stage_k(it), 16, 1024), idS);
                mma_commit_el(bs.st(0));
            };
            auto issue_dp = [&](int it) {  // dP = dO V^T
                mma_rows_by_rows<D>(bs.tmem + C::kColDP, ddO, sw128_desc(stage_k(it) + C::kTile, 16, 1024), idS);
                mma_commit_el(bs.st(1));
            };
            bool ok = bwait_warp(bs.bar_stat, 0, bs.abort_flag, p.status) &&
                      bwait_warp(bs.full(0), 0, bs.abort_flag, p.status);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
            }
            for (int it = 0; ok && it < T; ++it) {
                const uint32_t sk = stage_k(it);
                const bool more = it + 1 < T;
                if (!(ok = bwait_warp(bs.pp(0), it & 1, bs.abort_flag, p.status))) break;
                if (more) {
                    if (!(ok = bwait_warp(bs.full((it + 1) & 1), ((it + 1) >> 1) & 1, bs.abort_flag, p.status))) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
                if (!(ok = bwait_warp(bs.pp(1), it & 1, bs.abort_flag, p.status))) break;
                tc_fence_after();
                mma_tmem_by_tile(bs.tmem + C::kColAcc0, bs.tmem + C::kColDP, sw128_desc(sk, C::kChunk, 1024), idAcc,
                                 it == 0);  // dQ += dS K
                mma_commit_el(bs.empty(it & 1));  // K, V of this tile fully read
                if (more) issue_dp(it + 1);
            }
            if (ok) mma_commit_el(bs.bar_done);
            mma_commit_el(bs.bar_drain);
            bwait_warp_final(bs.bar_drain, 0, p.status);
        }
        __syncwarp();
    } else {
        // elementwise: thread = query row of the tile (TMEM lane); columns = keys
        const int r = (warp & 3) * 32 + lane, half = warp >> 2;  // row; column half of the tile
        const int row = i0 + r;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const float c = p.scale_log2;
        const float nlse2 = p.nlse2[(size_t)bh * p.Mpad + row];  // +inf past M (masked)
        const float ndel = p.ndelta[(size_t)bh * p.Mpad + row];
        const uint64_t c2 = f2_pack(c, c), nl2 = f2_pack(nlse2, nlse2), nd2 = f2_pack(ndel, ndel);
        const int pos = row + off;
        bool ok = true;
        for (int it = 0; ok && it < T; ++it) {
            const int k0 = (kt0 + (it + rot) % T) * BT;
            const bool need_mask = (i0 + BT > p.M) || (k0 + BT > p.N) ||
                                   (p.causal && k0 + BT - 1 > i0 + off) ||
                                   (p.window > 0 && k0 <= i0 + BT - 1 + off - p.window);
            // ---- phase A: P = exp2(S c - lse2), kept in registers ----
            if (!(ok = bwait_warp(bs.st(0), it & 1, bs.abort_flag, p.status))) break;
            tc_fence_after();
            uint32_t sva[2][32];
            tmem_ld_x32(bs.tmem + lane_base + C::kColS + 64 * half, sva[0]);
            tmem_ld_x32(bs.tmem + lane_base + C::kColS + 64 * half + 32, sva[1]);
            tmem_wait_ld_x32(sva[0]);
            reg_after_x32(sva[1]);
            // S is in registers: the next tile's score product may overwrite it
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(bs.pp(0));
            uint32_t pkeep[2][16];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int q4 = 2 * half + qq, c0 = q4 * 32;  // TMEM column = key of the tile
                const uint32_t* sv = sva[qq];
                // visible keys of this chunk for this thread's row: e in [elo, ehi)
                int elo = 0, ehi = 32;
                if (need_mask) {
                    const int kc = k0 + c0;  // key of e = 0
                    if (row >= p.M) ehi = 0;
                    ehi = min(ehi, p.N - kc);
                    if (p.causal) ehi = min(ehi, pos + 1 - kc);
                    if (p.window > 0) elo = max(elo, pos - p.window + 1 - kc);
                }
                uint32_t pk[16];
                auto chunk = [&](auto masked) {
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        float x[2], pr[2];
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e2]), __uint_as_float(sv[2 * e2 + 1])), c2, nl2),
                                  x[0], x[1]);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int e = 2 * e2 + u;
                            float pv = ex2(x[u]);
                            if (decltype(masked)::value) pv = (e >= elo && e < ehi) ? pv : 0.f;
                            pr[u] = pv;
                        }
                        pk[e2] = bpack2<kBF16>(pr[0], pr[1]);
                    }
                };
                if (need_mask)
                    chunk(std::true_type{});
                else
                    chunk(std::false_type{});
#pragma unroll
                for (int x = 0; x < 16; ++x) pkeep[qq][x] = pk[x];
            }
            // ---- phase B: dS = P (dP - delta), packed over dP ----
            if (!(ok = bwait_warp(bs.st(1), it & 1, bs.abort_flag, p.status))) break;
            tc_fence_after();
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const int q4 = 2 * half + qq, c0 = q4 * 32;
                uint32_t dpv[32];
                tmem_ld_x32(bs.tmem + lane_base + C::kColDP + c0, dpv);
                tmem_wait_ld_x32(dpv);
                const uint32_t* pv16 = pkeep[qq];
                uint32_t dk[16];
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    float p0, p1, y0, y1;
                    unpack2<kBF16>(pv16[e2], p0, p1);
                    f2_unpack(f2_mul(f2_pack(p0, p1),
                                     f2_add(f2_pack(__uint_as_float(dpv[2 * e2]), __uint_as_float(dpv[2 * e2 + 1])), nd2)),
                              y0, y1);
                    dk[e2] = bpack2<kBF16>(y0, y1);
                }
                tmem_st_x16(bs.tmem + lane_base + C::kColDP + packed_col(q4), dk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();  // the warp's TMEM stores before lane 0's arrival
            if ((threadIdx.x & 31) == 0) mbar_arrive(bs.pp(1));
        }
        uint16_t* dq_row = reinterpret_cast<uint16_t*>(p.out0) + ((size_t)bh * p.M + row) * D;
        const bool write = row < p.M;
        if (T == 0) {  // no key visible to any row of the tile: zero gradient
            if (write)
#pragma unroll
                for (int x = half * (D / 16); x < (half + 1) * (D / 16); ++x)
                    reinterpret_cast<uint4*>(dq_row)[x] = make_uint4(0, 0, 0, 0);
        } else {
            const uint32_t boxes = bs.sbase + C::kOffStage;
            if (ok && bwait_warp(bs.bar_done, 0, bs.abort_flag, p.status)) {
                tc_fence_after();
                stage_row<D, kBF16>(bs.tmem + lane_base + C::kColAcc0, p.scale, boxes, r, half);
                fence_proxy_async_smem();  // the boxes are read by the TMA (async proxy)
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bs.bar_ep);  // every warp arrives, also after giving up
            store_boxes<D>(bs, boxes, &tmdQ, &tmdQ, 1, i0, bh, p.status);
        }
    }
    bwd_teardown(bs);
    // This grid completes only after the dK/dV grid it may overlap has completed and its
    // writes are visible (its CTAs start while that grid's last wave runs).
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// dot product of eight 16-bit pairs held in two 16-byte vectors
template <bool kBF16>
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float a0, a1, b0, b1;
        if (kBF16) {
            a0 = __uint_as_float(wa[i] << 16);
            a1 = __uint_as_float(wa[i] & 0xFFFF0000u);
            b0 = __uint_as_float(wb[i] << 16);
            b1 = __uint_as_float(wb[i] & 0xFFFF0000u);
        } else {
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&wa[i]));
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&wb[i]));
            a0 = fa.x;
            a1 = fa.y;
            b0 = fb.x;
            b1 = fb.y;
        }
        acc = fmaf(a0, b0, acc);
        acc = fmaf(a1, b1, acc);
    }
    return acc;
}

// ndelta = -rowsum(dO * O) and nlse2 = -lse * log2(e) per row, padded to Mpad rows
// per head (+inf and 0 past M). D / 8 lanes per row, each with one 16-byte load
// of O and of dO, so a warp covers 32 / (D / 8) rows; the row sums reduce
// within each lane group.
template <bool kBF16, int D>
__global__ void __launch_bounds__(256)
    attn_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ d_o, const float* __restrict__ lse,
                        float* nlse2, float* ndelta, int M, int Mpad, int rows_pad) {
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int li = lane % kLanesPerRow;
    const int gr = (blockIdx.x * 8 + warp) * kRowsPerWarp + lane / kLanesPerRow;
    const bool valid = gr < rows_pad;
    const int bh = gr / Mpad, i = gr % Mpad;
    const size_t row = (size_t)bh * M + i;
    float acc = 0.f;
    if (valid && i < M)
        acc = dot8<kBF16>(reinterpret_cast<const uint4*>(o + row * D)[li],
                          reinterpret_cast<const uint4*>(d_o + row * D)[li]);
#pragma unroll
    for (int s = kLanesPerRow / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (valid && li == 0) {
        ndelta[gr] = i < M ? -acc : 0.f;
        nlse2[gr] = i < M ? -(lse[row] * kLog2e) : INFINITY;
    }
}

// ---------------------------------------------------------------------------
// CUDA-core backward for the small head dimensions (D = 16, 32): the same
// formulas and the same split (one kernel owns dK and dV of key rows, the other
// dQ of query rows; nothing is accumulated across blocks), one warp per output
// row, one lane per query row (dK/dV) or per key (dQ) of a 32-wide tile staged
// in shared memory as FP32. P and dS stay FP32 (no 16-bit rounding between the
// products): a correct covering path for the pages' own head dimensions.
// ---------------------------------------------------------------------------
struct SimtBwdArgs {
    const uint16_t *q, *k, *v, *d_o;
    const float* nlse2;   // [B*Hq][Mpad], from the pre kernel
    const float* ndelta;  // [B*Hq][Mpad]
    uint16_t *dq, *dk, *dv;
    int Hq, Hkv, M, N, G, Mpad;
    int causal, window;
    float scale, scale_log2;
};

constexpr int kSBRows = 16;  // output rows (warps) per block
constexpr int kSBTile = 32;  // staged rows per tile, one per lane

template <bool kBF16>
__device__ __forceinline__ float ld16(const uint16_t* p, size_t i) {
    const uint32_t x = p[i];
    return kBF16 ? __uint_as_float(x << 16) : __half2float(__ushort_as_half((unsigned short)x));
}
template <bool kBF16>
__device__ __forceinline__ uint16_t st16(float x) {
    return kBF16 ? __bfloat16_as_ushort(__float2bfloat16_rn(x)) : __half_as_ushort(__float2half_rn(x));
}

// dK, dV: block = kSBRows key rows of one KV head (grid: key-row blocks x B*Hkv).
// For every query head of the group and every 32-row query tile that may see
// the block's keys: lane = query row, p = exp2(s c - lse2), dp = dO . v,
// ds = p (dp - delta); dV += p dO, dK += ds Q (a shuffle sum over the lanes).
template <bool kBF16, int D>
__global__ void __launch_bounds__(kSBRows * 32) attn_bwd_simt_dkdv_kernel(const SimtBwdArgs a) {
    constexpr int EPL = (D + 31) / 32;
    __shared__ float qs[kSBTile][D + 1], dos[kSBTile][D + 1];
    __shared__ float kr[kSBRows][D], vr[kSBRows][D];
    __shared__ float l2s[kSBTile], dls[kSBTile];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = blockIdx.y, b = grp / a.Hkv, g = grp % a.Hkv;
    const int j0 = blockIdx.x * kSBRows, j = j0 + warp;
    const int jl = min(j0 + kSBRows, a.N) - 1;  // the block's last key
    const int off = a.N - a.M;                  // row i sits at key position i + off
    const size_t kvrow = (size_t)grp * a.N;
    for (int x = threadIdx.x; x < kSBRows * D; x += blockDim.x) {
        const int r = x / D, d = x % D;
        const bool in = j0 + r < a.N;
        kr[r][d] = in ? ld16<kBF16>(a.k, (kvrow + j0 + r) * D + d) : 0.f;
        vr[r][d] = in ? ld16<kBF16>(a.v, (kvrow + j0 + r) * D + d) : 0.f;
    }
    // query rows that may see any of the block's keys
    int i_lo = 0, i_hi = a.M;
    if (a.causal) i_lo = max(0, j0 - off);
    if (a.window > 0) i_hi = min(a.M, jl + a.window - off);
    float ak[EPL], av[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) ak[e] = av[e] = 0.f;
    for (int hh = 0; hh < a.G; ++hh) {
        const int bh = b * a.Hq + g * a.G + hh;
        for (int i0 = i_lo; i0 < i_hi; i0 += kSBTile) {
            __syncthreads();  // the previous tile consumed (and kr, vr written)
            for (int x = threadIdx.x; x < kSBTile * D; x += blockDim.x) {
                const int r = x / D, d = x % D, i = i0 + r;
                const bool in = i < i_hi;
                qs[r][d] = in ? ld16<kBF16>(a.q, ((size_t)bh * a.M + i) * D + d) : 0.f;
                dos[r][d] = in ? ld16<kBF16>(a.d_o, ((size_t)bh * a.M + i) * D + d) : 0.f;
            }
            if (threadIdx.x < kSBTile) {
                const int i = i0 + threadIdx.x;
                l2s[threadIdx.x] = i < i_hi ? a.nlse2[(size_t)bh * a.Mpad + i] : 0.f;
                dls[threadIdx.x] = i < i_hi ? a.ndelta[(size_t)bh * a.Mpad + i] : 0.f;
            }
            __syncthreads();
            if (j < a.N) {
                const int i = i0 + lane;
                int lo = 0, hi = 0;
                if (i < i_hi) key_range(i + off, a.N, a.causal, a.window, &lo, &hi);
                float p = 0.f, ds = 0.f;
                if (j >= lo && j < hi) {
                    float s = 0.f, dp = 0.f;
#pragma unroll
                    for (int d = 0; d < D; ++d) {
                        s = fmaf(qs[lane][d], kr[warp][d], s);
                        dp = fmaf(dos[lane][d], vr[warp][d], dp);
                    }
                    p = exp2f(fmaf(s, a.scale_log2, l2s[lane]));
                    ds = p * (dp + dls[lane]);
                }
#pragma unroll 4
                for (int ii = 0; ii < kSBTile; ++ii) {
                    const float pi = __shfl_sync(0xffffffffu, p, ii), dsi = __shfl_sync(0xffffffffu, ds, ii);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) {
                        const int d = lane + 32 * e;
                        if (d < D) {
                            av[e] = fmaf(pi, dos[ii][d], av[e]);
                            ak[e] = fmaf(dsi, qs[ii][d], ak[e]);
                        }
                    }
                }
            }
        }
    }
    if (j >= a.N) return;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const int d = lane + 32 * e;
        if (d < D) {
            a.dk[(kvrow + j) * D + d] = st16<kBF16>(ak[e] * a.scale);
            a.dv[(kvrow + j) * D + d] = st16<kBF16>(av[e]);
        }
    }
}

// dQ: block = kSBRows query rows of one query head (grid: row blocks x B*Hq);
// lane = key of a 32-key tile over the keys the block's rows may see.
template <bool kBF16, int D>
__global__ void __launch_bounds__(kSBRows * 32) attn_bwd_simt_dq_kernel(const SimtBwdArgs a) {
    constexpr int EPL = (D + 31) / 32;
    __shared__ float ks[kSBTile][D + 1], vs[kSBTile][D + 1];
    __shared__ float qr[kSBRows][D], dor[kSBRows][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.y, b = bh / a.Hq, h = bh % a.Hq;
    const size_t kvrow = ((size_t)b * a.Hkv + h / a.G) * a.N;
    const int r0 = blockIdx.x * kSBRows, i = r0 + warp;
    const int rl = min(r0 + kSBRows, a.M) - 1;
    const int off = a.N - a.M;
    for (int x = threadIdx.x; x < kSBRows * D; x += blockDim.x) {
        const int r = x / D, d = x % D;
        const bool in = r0 + r < a.M;
        qr[r][d] = in ? ld16<kBF16>(a.q, ((size_t)bh * a.M + r0 + r) * D + d) : 0.f;
        dor[r][d] = in ? ld16<kBF16>(a.d_o, ((size_t)bh * a.M + r0 + r) * D + d) : 0.f;
    }
    // keys any row of the block may see (both bounds grow with the position)
    int lo_f, hi_f, lo_l, hi_l;
    key_range(r0 + off, a.N, a.causal, a.window, &lo_f, &hi_f);
    key_range(rl + off, a.N, a.causal, a.window, &lo_l, &hi_l);
    int r_lo = 0, r_hi = 0;
    float nl2 = 0.f, nd = 0.f;
    if (i < a.M) {
        key_range(i + off, a.N, a.causal, a.window, &r_lo, &r_hi);
        nl2 = a.nlse2[(size_t)bh * a.Mpad + i];
        nd = a.ndelta[(size_t)bh * a.Mpad + i];
    }
    float aq[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) aq[e] = 0.f;
    for (int t0 = lo_f; t0 < hi_l; t0 += kSBTile) {
        __syncthreads();
        for (int x = threadIdx.x; x < kSBTile * D; x += blockDim.x) {
            const int r = x / D, d = x % D, jj = t0 + r;
            const bool in = jj < hi_l;
            ks[r][d] = in ? ld16<kBF16>(a.k, (kvrow + jj) * D + d) : 0.f;
            vs[r][d] = in ? ld16<kBF16>(a.v, (kvrow + jj) * D + d) : 0.f;
        }
        __syncthreads();
        if (i < a.M) {
            const int jj = t0 + lane;
            float ds = 0.f;
            if (jj >= r_lo && jj < r_hi) {
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int d = 0; d < D; ++d) {
                    s = fmaf(qr[warp][d], ks[lane][d], s);
                    dp = fmaf(dor[warp][d], vs[lane][d], dp);
                }
                const float p = exp2f(fmaf(s, a.scale_log2, nl2));
                ds = p * (dp + nd);
            }
#pragma unroll 4
            for (int u = 0; u < kSBTile; ++u) {
                const float dsu = __shfl_sync(0xffffffffu, ds, u);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const int d = lane + 32 * e;
                    if (d < D) aq[e] = fmaf(dsu, ks[u][d], aq[e]);
                }
            }
        }
    }
    if (i >= a.M) return;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const int d = lane + 32 * e;
        if (d < D) a.dq[((size_t)bh * a.M + i) * D + d] = st16<kBF16>(aq[e] * a.scale);
    }
}

template <int D, bool kBF16>
cudaError_t launch_bwd_simt_t(const Problem& pr, const BwdArgs& a, const float* lse2, const float* delta, int Mpad,
                              cudaStream_t stream) {
    const int rows_pad = pr.B * pr.Hq * Mpad;
    constexpr int kPreRowsPerBlock = 8 * (32 / (D / 8));
    attn_bwd_pre_kernel<kBF16, D><<<(rows_pad + kPreRowsPerBlock - 1) / kPreRowsPerBlock, 256, 0, stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.d_o), a.lse, const_cast<float*>(lse2),
        const_cast<float*>(delta), pr.M, Mpad, rows_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    SimtBwdArgs sa;
    sa.q = static_cast<const uint16_t*>(a.q);
    sa.k = static_cast<const uint16_t*>(a.k);
    sa.v = static_cast<const uint16_t*>(a.v);
    sa.d_o = static_cast<const uint16_t*>(a.d_o);
    sa.nlse2 = lse2;
    sa.ndelta = delta;
    sa.dq = static_cast<uint16_t*>(a.dq);
    sa.dk = static_cast<uint16_t*>(a.dk);
    sa.dv = static_cast<uint16_t*>(a.dv);
    sa.Hq = pr.Hq;
    sa.Hkv = pr.Hkv;
    sa.M = pr.M;
    sa.N = pr.N;
    sa.G = pr.G;
    sa.Mpad = Mpad;
    sa.causal = pr.causal;
    sa.window = pr.window;
    sa.scale = pr.scale;
    sa.scale_log2 = pr.scale_log2;
    attn_bwd_simt_dkdv_kernel<kBF16, D>
        <<<dim3((pr.N + kSBRows - 1) / kSBRows, pr.B * pr.Hkv), kSBRows * 32, 0, stream>>>(sa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    attn_bwd_simt_dq_kernel<kBF16, D>
        <<<dim3((pr.M + kSBRows - 1) / kSBRows, pr.B * pr.Hq), kSBRows * 32, 0, stream>>>(sa);
    return cudaGetLastError();
}

template <int D, bool kBF16>
cudaError_t launch_bwd_t(const Problem& pr, const BwdArgs& a, const float* lse2, const float* delta, int Mpad,
                         int* status, cudaStream_t stream) {
    using C = BCfg<D>;
    static PerDeviceOnce attr_once;
    const cudaError_t attr_err = once_per_device(attr_once, [] {
        cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, kBF16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::kSmem);
        return e;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int rows_pad = pr.B * pr.Hq * Mpad;
    constexpr int kPreRowsPerBlock = 8 * (32 / (D / 8));
    attn_bwd_pre_kernel<kBF16, D><<<(rows_pad + kPreRowsPerBlock - 1) / kPreRowsPerBlock, 256, 0, stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.d_o), a.lse, const_cast<float*>(lse2),
        const_cast<float*>(delta), pr.M, Mpad, rows_pad);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
    if (!make_tensor_map(&tq, a.q, D, pr.M, pr.B * pr.Hq, BT, kBF16) ||
        !make_tensor_map(&tdo, a.d_o, D, pr.M, pr.B * pr.Hq, BT, kBF16) ||
        !make_tensor_map(&tk, a.k, D, pr.N, pr.B * pr.Hkv, BT, kBF16) ||
        !make_tensor_map(&tv, a.v, D, pr.N, pr.B * pr.Hkv, BT, kBF16) ||
        !make_tensor_map(&tdq, a.dq, D, pr.M, pr.B * pr.Hq, BT, kBF16) ||
        !make_tensor_map(&tdk, a.dk, D, pr.N, pr.B * pr.Hkv, BT, kBF16) ||
        !make_tensor_map(&tdv, a.dv, D, pr.N, pr.B * pr.Hkv, BT, kBF16))
        return cudaErrorInvalidValue;
    BwdParams bp = {};
    bp.nlse2 = lse2;
    bp.ndelta = delta;
    bp.status = status;
    bp.Hq = pr.Hq;
    bp.Hkv = pr.Hkv;
    bp.M = pr.M;
    bp.N = pr.N;
    bp.G = pr.G;
    bp.Mpad = Mpad;
    bp.causal = pr.causal;
    bp.window = pr.window;
    bp.scale = pr.scale;
    bp.scale_log2 = pr.scale_log2;
    // dK, dV
    bp.out0 = a.dk;
    bp.out1 = a.dv;
    bp.groups = pr.B * pr.Hkv;
    bp.ntile = (pr.N + BT - 1) / BT;
    attn_bwd_dkdv_kernel<D, kBF16><<<bp.groups * bp.ntile, kBwdThreads, C::kSmem, stream>>>(tq, tk, tv, tdo, tdk,
                                                                                           tdv, bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // dQ
    bp.out0 = a.dq;
    bp.out1 = nullptr;
    bp.groups = pr.B * pr.Hq;
    bp.ntile = (pr.M + BT - 1) / BT;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(bp.groups * bp.ntile);
    cfg.blockDim = dim3(kBwdThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_bwd_dq_kernel<D, kBF16>, tq, tk, tv, tdo, tdq, bp);
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int M) {
    const size_t Mpad = ((size_t)M + BT - 1) / BT * BT;
    const size_t part = ((size_t)B * Hq * Mpad * sizeof(float) + 255) & ~(size_t)255;
    return 2 * part;
}

cudaError_t launch_bwd(const Problem& p, const BwdArgs& a, void* ws, int* status, cudaStream_t stream) {
    const int Mpad = (p.M + BT - 1) / BT * BT;
    const size_t part = ((size_t)p.B * p.Hq * Mpad * sizeof(float) + 255) & ~(size_t)255;
    const float* lse2 = static_cast<const float*>(ws);
    const float* delta = reinterpret_cast<const float*>(static_cast<const char*>(ws) + part);
    const bool bf = p.dtype == ATTN_BF16;
    if (p.D == 128)
        return bf ? launch_bwd_t<128, true>(p, a, lse2, delta, Mpad, status, stream)
                  : launch_bwd_t<128, false>(p, a, lse2, delta, Mpad, status, stream);
    if (p.D == 64)
        return bf ? launch_bwd_t<64, true>(p, a, lse2, delta, Mpad, status, stream)
                  : launch_bwd_t<64, false>(p, a, lse2, delta, Mpad, status, stream);
    if (p.D == 32)
        return bf ? launch_bwd_simt_t<32, true>(p, a, lse2, delta, Mpad, stream)
                  : launch_bwd_simt_t<32, false>(p, a, lse2, delta, Mpad, stream);
    if (p.D == 16)
        return bf ? launch_bwd_simt_t<16, true>(p, a, lse2, delta, Mpad, stream)
                  : launch_bwd_simt_t<16, false>(p, a, lse2, delta, Mpad, stream);
    return cudaErrorInvalidValue;
}

}  // namespace attn
