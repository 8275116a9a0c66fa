// Prefill forward with the pair MMA (tcgen05 cta_group::2), sm_103a, D = 128,
// 16-bit inputs.
//
// A thread-block cluster of two CTAs (one per SM) shares each work tile of 512
// query rows of one (batch, head). The ping query tile A is rows [r, r + 256) and
// the pong tile B rows [r + 256, r + 512); CTA k holds rows r + 128 k .. of A and
// r + 256 + 128 k .. of B in its own shared memory, and its 128 rows of every
// score and output tile live in its own TMEM. One thread of CTA 0 (the leader)
// issues every MMA with M = 256: the pair instruction takes A's rows from both
// CTAs' shared memory or TMEM at the same address, the first half of B's N
// columns from CTA 0 and the second half from CTA 1, and writes each CTA's rows of
// D into that CTA's TMEM. So each CTA loads half of every key tile (64 keys, the
// score product's N) and half of every value tile (64 output columns, the value
// product's N): per SM, half the K/V bytes and half the B-operand shared-memory
// reads of the one-CTA kernel, for the same MMA work.
//
// Warp roles per CTA: 0-3 softmax + epilogue of tile A's rows, 4-7 of tile B's,
// 8 TMA producer (this CTA's halves), 9 the MMA issuer in CTA 0 and, in CTA 1,
// the relay that forwards the completion of each of CTA 1's loads to CTA 0's
// barrier (a remote arrival), so the leader waits on one barrier per load.
// Commits go to both CTAs' barriers (multicast); the softmax warps of CTA 1
// arrive on CTA 0's P-ready and O-free barriers through distributed shared memory.
// TMEM (512 columns in each CTA, allocated by one warp of each CTA together):
// S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512); P over S.
//
// The softmax, lazy rescale, masking and epilogue are those of the one-CTA
// kernel (each CTA handles its own rows). Every wait is bounded (1 s); on expiry
// a CTA raises its abort flag, sets the device status word and leaves its loops;
// both CTAs drain their copies and MMAs and meet at a final cluster barrier
// before TMEM is freed.
#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "tma_map.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int PD = 128;                 // head dimension
constexpr int PBM = 128;                // rows of a query tile per CTA
constexpr int PBN = 128;                // keys per key tile
constexpr int PNQ = 2;                  // query tiles (A, B) per work tile
constexpr int PRows = 2 * PNQ * PBM;    // rows per work tile: 512
constexpr int kPThreads = 320;
constexpr int kPLoadWarp = 8, kPMmaWarp = 9;
constexpr uint64_t kPTimeoutNs = 1000000000ull;
constexpr float kPRescaleThreshold = 8.0f;

// Shared memory of one CTA
constexpr int kPQTile = PBM * PD * 2;          // 32 KB: 128 rows x 128 columns
constexpr int kPQChunk = PBM * 128;            // 16 KB: one 64-column chunk of a Q tile
constexpr int kPSlot = 16384;                  // a ring slot: K half (64 keys x 128) or V half (128 keys x 64)
constexpr int kPKChunk = 64 * 128;             // 8 KB: one 64-column chunk of a K half
constexpr int kPStages = 8;
constexpr int kPHalf = kPStages / 2;
constexpr int kPQOff = 0;
constexpr int kPKVOff = PNQ * kPQTile;                   // 64 KB
constexpr int kPStageOff = kPKVOff + kPStages * kPSlot;  // 192 KB: epilogue staging, 4 KB per softmax warp
constexpr int kPBarOff = kPStageOff + 8 * 4096;          // 224 KB
// q_full, q_free, full[8], empty[8], s_full[2], p_full[2], o_final, o_free[2], drain
constexpr int kPNumBars = 2 + 2 * kPStages + 2 + 2 + 1 + 2 + 1;
constexpr int kPMiscOff = kPBarOff + 8 * kPNumBars;
constexpr int kPSmemBytes = kPMiscOff + 16 + 1024;

__host__ __device__ constexpr uint32_t pcol_s(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t pcol_o(int t) { return t ? 384u : 256u; }

struct PairParams {
    void* o;
    float* lse;
    int* status;
    int M, N, Hq, Hkv, G;
    int causal, window;
    float scale_log2;
    int BH;     // B * Hq
    int nqb;    // work tiles per head: ceil(M / 512)
    int tiles;  // BH * nqb
};

struct PBars {
    uint32_t q_full, q_free, full0, empty0, s0, p0, o_final, o_free0, drain;
    __device__ uint32_t full(int s) const { return full0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return empty0 + 8u * s; }
    __device__ uint32_t s_full(int t) const { return s0 + 8u * t; }
    __device__ uint32_t p_full(int t) const { return p0 + 8u * t; }
    __device__ uint32_t o_free(int t) const { return o_free0 + 8u * t; }
};

struct PWork {
    int bh, kvh, row0, jt0, n;
};

// w-th work tile of this pair (serpentine over a longest-first order); false when done
__device__ __forceinline__ bool pair_work_tile(const PairParams& p, int w, PWork* t) {
    const int pairs = gridDim.x >> 1, c = blockIdx.x >> 1;
    const int idx = w * pairs + ((w & 1) ? pairs - 1 - c : c);
    if (idx >= p.tiles) return false;
    const int qb = p.nqb - 1 - idx / p.BH;
    t->bh = idx % p.BH;
    const int b = t->bh / p.Hq, h = t->bh % p.Hq;
    t->kvh = b * p.Hkv + h / p.G;
    t->row0 = qb * PRows;
    const int off = p.N - p.M;
    const int last_row = min(t->row0 + PRows - 1, p.M - 1);
    int klo = 0, khi = p.N, unused = 0;
    key_range(t->row0 + off, p.N, p.causal, p.window, &klo, &unused);
    key_range(last_row + off, p.N, p.causal, p.window, &unused, &khi);
    t->jt0 = klo / PBN;
    t->n = (khi > klo) ? (khi + PBN - 1) / PBN - t->jt0 : 0;
    return true;
}

// first row of query tile t of work tile `row0` held by cluster CTA `rank`
__device__ __forceinline__ int pair_tile_row(int row0, int t, int rank) { return row0 + t * 2 * PBM + rank * PBM; }

__device__ __forceinline__ uint32_t p_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t p_map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void p_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// arrival on a barrier of a cluster CTA (shared::cluster address), release at cluster scope
__device__ __forceinline__ void p_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// true once the phase with this parity completed, acquiring at cluster scope
__device__ __forceinline__ bool p_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool p_test_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// pair forms of the TMEM allocation, the MMA and the commit (to both CTAs' barriers)
__device__ __forceinline__ void p_tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void p_tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void p_tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void p_mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void p_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void p_commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"((uint16_t)3)
        : "memory");
}

// bounded single-thread wait (cluster-scope acquire)
__device__ bool pwait_one(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status,
                          bool abortable = true) {
    if (p_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (p_try_wait_cluster(bar, parity)) return true;
        if (abortable && *abort_flag) return false;
        if (globaltimer_ns() - t0 > kPTimeoutNs) {
            *abort_flag = 1u;
            atomicExch(status, 1);
            return false;
        }
    }
}
// bounded warp-uniform wait
__device__ bool pwait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        const bool done = p_try_wait_cluster(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        int stop = 0;
        if (lane == 0) {
            if (*abort_flag) {
                stop = 1;
            } else if (globaltimer_ns() - t0 > kPTimeoutNs) {
                *abort_flag = 1u;
                atomicExch(status, 1);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

template <bool kBF16>
__device__ __forceinline__ uint32_t ppack2(float lo, float hi) {
    return kBF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

// S_t = Q_t K_j^T over D = 128: eight K steps of 16; A is a 128-row Q tile
// (16 KB per 64-column chunk), B a 64-row K half (8 KB per chunk)
__device__ __forceinline__ void pair_group_s(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < PD / 16; ++kk) {
        const uint64_t ao = (uint64_t)((((kk >> 2) * kPQChunk) + (kk & 3) * 32) >> 4);
        const uint64_t bo = (uint64_t)((((kk >> 2) * kPKChunk) + (kk & 3) * 32) >> 4);
        p_mma_ss(d_tmem, a0 + ao, b0 + bo, idesc, kk > 0 ? 1u : 0u);
    }
}
// the same with `between` run after the first half of the K steps
template <class F>
__device__ __forceinline__ void pair_group_s(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc,
                                             F&& between) {
#pragma unroll
    for (int kk = 0; kk < PD / 16; ++kk) {
        if (kk == PD / 32) between();
        const uint64_t ao = (uint64_t)((((kk >> 2) * kPQChunk) + (kk & 3) * 32) >> 4);
        const uint64_t bo = (uint64_t)((((kk >> 2) * kPKChunk) + (kk & 3) * 32) >> 4);
        p_mma_ss(d_tmem, a0 + ao, b0 + bo, idesc, kk > 0 ? 1u : 0u);
    }
}
// O_t += P_t V_j: P from TMEM (8 columns per 16 keys), B a 128-key V half read
// MN-major (one 128-byte chunk per key; a K step is 16 key rows)
__device__ __forceinline__ void pair_group_pv(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, uint32_t idesc,
                                              bool first) {
#pragma unroll
    for (int kk = 0; kk < PBN / 16; ++kk)
        p_mma_ts(d_tmem, a_tmem + kk * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4), idesc,
                 (first && kk == 0) ? 0u : 1u);
}

template <bool kBF16>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const PairParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + kPQOff;
    const uint32_t sKV = sbase + kPKVOff;
    const uint32_t sStage = sbase + kPStageOff;
    PBars bar;
    bar.q_full = sbase + kPBarOff;
    bar.q_free = bar.q_full + 8;
    bar.full0 = bar.q_free + 8;
    bar.empty0 = bar.full0 + 8 * kPStages;
    bar.s0 = bar.empty0 + 8 * kPStages;
    bar.p0 = bar.s0 + 16;
    bar.o_final = bar.p0 + 16;
    bar.o_free0 = bar.o_final + 8;
    bar.drain = bar.o_free0 + 16;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + kPMiscOff);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = p_cluster_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        // the leader's load barriers take one more arrival: CTA 1's relay
        mbar_init(bar.q_full, leader ? 2 : 1);
        mbar_init(bar.q_free, 1);
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(bar.full(s), leader ? 2 : 1);
            mbar_init(bar.empty(s), 1);
        }
        for (int t = 0; t < PNQ; ++t) {
            mbar_init(bar.s_full(t), 1);
            mbar_init(bar.p_full(t), 8);  // one arrival per softmax warp of both CTAs (leader's barrier)
            mbar_init(bar.o_free(t), 8);
        }
        mbar_init(bar.o_final, 1);
        mbar_init(bar.drain, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == kPMmaWarp) {
        p_tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), 512);
        p_tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    p_cluster_sync();  // both CTAs' barriers and TMEM exist before any remote arrival or pair MMA
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kPLoadWarp) {
        // ---------------- TMA producer: this CTA's Q tiles and K/V halves ----------------
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            int u = 0, tc = 0, q_issued = 0;
            bool ok = true;
            PWork wk;
            for (int w = 0; ok && pair_work_tile(p, w, &wk); ++w) {
                if (wk.n == 0) continue;
                if (tc > 0 && !(ok = pwait_one(bar.q_free, (tc - 1) & 1, abort_flag, p.status))) break;
                mbar_arrive_expect_tx(bar.q_full, PNQ * kPQTile);
                for (int t = 0; t < PNQ; ++t)
                    for (int c = 0; c < 2; ++c)
                        tma_load_3d(sQ + t * kPQTile + c * kPQChunk, &tmQ, c * 64, pair_tile_row(wk.row0, t, rank),
                                    wk.bh, bar.q_full);
                ++q_issued;
                for (int x = 0; x < 2 * wk.n; ++x, ++u) {
                    const int s = u % kPStages;
                    // one commit after S_B(J) frees K_J and V_(J-1) (barrier J % kPHalf)
                    const int J = u >> 1;
                    const int Jf = (u & 1) ? J - kPHalf + 1 : J - kPHalf;
                    if (u >= kPStages &&
                        !(ok = pwait_one(bar.empty(Jf % kPHalf), (Jf / kPHalf) & 1, abort_flag, p.status)))
                        break;
                    mbar_arrive_expect_tx(bar.full(s), kPSlot);
                    const int key0 = (wk.jt0 + x / 2) * PBN;
                    if ((x & 1) == 0) {  // K: this CTA's 64 keys, both 64-column chunks
                        for (int c = 0; c < 2; ++c)
                            tma_load_3d(sKV + s * kPSlot + c * kPKChunk, &tmK, c * 64, key0 + 64 * (int)rank, wk.kvh,
                                        bar.full(s));
                    } else {  // V: all 128 keys, this CTA's 64 output columns
                        tma_load_3d(sKV + s * kPSlot, &tmV, 64 * (int)rank, key0, wk.kvh, bar.full(s));
                    }
                }
                ++tc;
            }
            if (q_issued > 0) pwait_one(bar.q_full, (q_issued - 1) & 1, abort_flag, p.status, false);
            for (int x = max(0, u - kPStages); x < u; ++x)
                pwait_one(bar.full(x % kPStages), (x / kPStages) & 1, abort_flag, p.status, false);
        }
    } else if (warp == kPMmaWarp && !leader) {
        // ---------------- relay (CTA 1): each of this CTA's loads, once landed, to the leader ----------------
        if (lane == 0) {
            const uint32_t rq = p_map_rank(bar.q_full, 0);
            int u = 0, tc = 0;
            bool ok = true;
            PWork wk;
            for (int w = 0; ok && pair_work_tile(p, w, &wk); ++w) {
                if (wk.n == 0) continue;
                if (!(ok = pwait_one(bar.q_full, tc & 1, abort_flag, p.status))) break;
                p_arrive_remote(rq);
                for (int x = 0; x < 2 * wk.n; ++x, ++u) {
                    const int s = u % kPStages;
                    if (!(ok = pwait_one(bar.full(s), (u / kPStages) & 1, abort_flag, p.status))) break;
                    p_arrive_remote(p_map_rank(bar.full(s), 0));
                }
                ++tc;
            }
        }
    } else if (warp == kPMmaWarp) {
        // ---------------- MMA issuer (CTA 0): M = 256 pair products ----------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f16(kBF16, 2 * PBM, PBN, false);
            constexpr uint32_t idPV = idesc_f16(kBF16, 2 * PBM, PD, true);
            int u = 0, tc = 0;
            int ps[PNQ] = {0, 0};
            bool ok = true;
            const uint64_t dq0 = sw128_desc(sQ, 16, 1024);
            const uint64_t dq1 = sw128_desc(sQ + kPQTile, 16, 1024);
            const uint64_t dk = sw128_desc(sKV, 16, 1024);
            const uint64_t dv = sw128_desc(sKV, kPSlot, 1024);  // one 64-column chunk per CTA: LBO unused
            constexpr uint64_t kSlotStep = (uint64_t)(kPSlot >> 4);
            bool p_ready = false;
            auto issue_pv = [&](int t, int slot, bool first) {
                if (!(t == 0 && p_ready) && !pwait_one(bar.p_full(t), ps[t] & 1, abort_flag, p.status)) return false;
                ++ps[t];
                if (first && tc > 0 && !pwait_one(bar.o_free(t), (tc - 1) & 1, abort_flag, p.status)) return false;
                tc_fence_after();
                pair_group_pv(tmem + pcol_o(t), tmem + pcol_s(t), dv + (uint64_t)slot * kSlotStep, idPV, first);
                return true;
            };
            PWork wk;
            for (int w = 0; ok && pair_work_tile(p, w, &wk); ++w) {
                const int n = wk.n;
                if (n == 0) continue;
                if (!(ok = pwait_one(bar.q_full, tc & 1, abort_flag, p.status))) break;
                tc_fence_after();
                int slot_v_prev = 0;
                for (int jj = 0; jj < n; ++jj) {
                    const int uk = u++, sk = uk % kPStages;
                    const int uv = u++, sv = uv % kPStages;
                    if (!(ok = pwait_one(bar.full(sk), (uk / kPStages) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    pair_group_s(tmem + pcol_s(0), dq0, dk + (uint64_t)sk * kSlotStep, idS);
                    p_commit_both(bar.s_full(0));
                    if (jj > 0 && !(ok = issue_pv(1, slot_v_prev, jj - 1 == 0))) break;
                    bool v_ready = false;
                    p_ready = false;
                    pair_group_s(tmem + pcol_s(1), dq1, dk + (uint64_t)sk * kSlotStep, idS, [&] {
                        v_ready = p_test_cluster(bar.full(sv), (uv / kPStages) & 1);
                        p_ready = p_test_cluster(bar.p_full(0), ps[0] & 1);
                    });
                    p_commit_both(bar.s_full(1));
                    if (jj == n - 1) p_commit_both(bar.q_free);
                    p_commit_both(bar.empty((uk >> 1) % kPHalf));  // K_j and V_(j-1) are read
                    if (!v_ready && !(ok = pwait_one(bar.full(sv), (uv / kPStages) & 1, abort_flag, p.status))) break;
                    if (!(ok = issue_pv(0, sv, jj == 0))) break;
                    slot_v_prev = sv;
                }
                if (!ok) break;
                if (!(ok = issue_pv(1, slot_v_prev, n - 1 == 0))) break;
                p_commit_both(bar.o_final);
                ++tc;
            }
            // all MMAs done (in both CTAs) before TMEM and shared memory are released
            p_commit_both(bar.drain);
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps (this CTA's rows) ----------------
        const int t = warp >> 2;
        const int wq = warp & 3;
        const int r_in_tile = wq * 32 + lane;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + pcol_s(t);
        const uint32_t tO = tmem + lane_base + pcol_o(t);
        const uint32_t rp = p_map_rank(bar.p_full(t), 0), ro = p_map_rank(bar.o_free(t), 0);
        const float c = p.scale_log2;
        const float masked_s = c >= 0.f ? -INFINITY : INFINITY;
        const int off = p.N - p.M;
        int g = 0, tc = 0;
        bool ok = true;
        PWork wk;
        for (int w = 0; ok && pair_work_tile(p, w, &wk); ++w) {
            const int tile_row0 = pair_tile_row(wk.row0, t, rank);
            const int row = tile_row0 + r_in_tile;
            if (wk.n == 0) {  // no row of this work tile sees any key: output 0
                if (row < p.M) {
                    if (p.lse) p.lse[(size_t)wk.bh * p.M + row] = -INFINITY;
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) +
                                                          ((size_t)wk.bh * p.M + row) * PD);
#pragma unroll
                    for (int v4 = 0; v4 < PD / 8; ++v4) dst[v4] = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            const int pos = row + off;
            const int tile_first_pos = tile_row0 + off;
            const int tile_last_pos = tile_first_pos + PBM - 1;
            float m_ref = -INFINITY;
            float l = 0.f;
            for (int jj = 0; jj < wk.n; ++jj, ++g) {
                const int key0 = (wk.jt0 + jj) * PBN;
                if (!(ok = pwait_warp(bar.s_full(t), g & 1, abort_flag, p.status))) break;
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) tmem_ld_x32(tS + q4 * 32, s[q4]);
                tmem_wait_ld_x32(s[0]);
                reg_after_x32(s[1]);
                reg_after_x32(s[2]);
                reg_after_x32(s[3]);
                const bool need_mask = (key0 + PBN > p.N) || (p.causal && key0 + PBN - 1 > tile_first_pos) ||
                                       (p.window > 0 && key0 <= tile_last_pos - p.window);
                if (need_mask) {
                    int lo = 0, hi = 0;
                    key_range(pos, p.N, p.causal, p.window, &lo, &hi);
                    const int vlo = lo - key0, vhi = hi - key0;
                    if (p.window > 0) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (q4 * 32 + e < vlo || q4 * 32 + e >= vhi) s[q4][e] = __float_as_uint(masked_s);
                    } else {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (q4 * 32 + e >= vhi) s[q4][e] = __float_as_uint(masked_s);
                    }
                }
                float mx;
                {
#define SV(i) __uint_as_float(s[(i) >> 5][(i) & 31])
                    float a0 = SV(0), a1 = SV(1), a2 = SV(2), a3 = SV(3);
                    if (c >= 0.f) {
#pragma unroll
                        for (int i = 4; i < 128; i += 8) {
                            a0 = max3f(a0, SV(i), SV(i + 1));
                            a1 = max3f(a1, SV(i + 2), SV(i + 3));
                            if (i + 4 < 128) {
                                a2 = max3f(a2, SV(i + 4), SV(i + 5));
                                a3 = max3f(a3, SV(i + 6), SV(i + 7));
                            }
                        }
                        mx = max3f(a0, a1, fmaxf(a2, a3));
                    } else {
#pragma unroll
                        for (int i = 4; i < 128; i += 8) {
                            a0 = min3f(a0, SV(i), SV(i + 1));
                            a1 = min3f(a1, SV(i + 2), SV(i + 3));
                            if (i + 4 < 128) {
                                a2 = min3f(a2, SV(i + 4), SV(i + 5));
                                a3 = min3f(a3, SV(i + 6), SV(i + 7));
                            }
                        }
                        mx = min3f(a0, a1, fminf(a2, a3));
                    }
#undef SV
                }
                const float m_tile = mx * c;
                const float m_new = fmaxf(m_ref, m_tile);
                const bool need = m_new > m_ref + kPRescaleThreshold;
                float alpha = 1.f;
                if (need) {
                    alpha = ex2(m_ref - m_new);
                    l *= alpha;
                    m_ref = m_new;
                }
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_use, -m_use);
                uint64_t lsum[2] = {0ull, 0ull};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t packed[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[q4][2 * e]), __uint_as_float(s[q4][2 * e + 1])), c2,
                                         nm2),
                                  x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        lsum[e & 1] = f2_add(lsum[e & 1], f2_pack(p0, p1));
                        packed[e] = ppack2<kBF16>(p0, p1);
                    }
                    tmem_st_x16(tS + q4 * 16, packed);
                }
                {
                    float l0, l1, l2, l3;
                    f2_unpack(lsum[0], l0, l1);
                    f2_unpack(lsum[1], l2, l3);
                    l += (l0 + l1) + (l2 + l3);
                }
                // rescale the accumulator (the previous value product completed: its commit
                // preceded this tile's score commit)
                if (__any_sync(0xffffffffu, need) && jj > 0) {
                    const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                    for (int ch = 0; ch < PD / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld_x32(tO + ch * 32, o);
                        tmem_wait_ld_x32(o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float y0, y1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), a2),
                                      y0, y1);
                            o[2 * e] = __float_as_uint(y0);
                            o[2 * e + 1] = __float_as_uint(y1);
                        }
                        tmem_st_x32(tO + ch * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) p_arrive_remote(rp);  // P ready: one arrival per warp on the leader's barrier
            }
            if (!ok) break;

            // ---------------- epilogue: O / l, one cast, rows < M (as in the one-CTA kernel) ----------------
            if (!(ok = pwait_warp(bar.o_final, tc & 1, abort_flag, p.status))) break;
            ++tc;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (p.lse && row < p.M)
                p.lse[(size_t)wk.bh * p.M + row] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
            const uint32_t wst = sStage + (t * 4 + wq) * 4096;
            const uint64_t inv2 = f2_pack(inv, inv);
            char* obase = reinterpret_cast<char*>(p.o) + ((size_t)wk.bh * p.M + tile_row0 + wq * 32) * (PD * 2);
            const int rows_left = p.M - (tile_row0 + wq * 32);
#pragma unroll
            for (int h = 0; h < PD / 64; ++h) {
                uint32_t o[2][32];
                tmem_ld_x32(tO + h * 64, o[0]);
                tmem_ld_x32(tO + h * 64 + 32, o[1]);
                tmem_wait_ld_x32(o[0]);
                reg_after_x32(o[1]);
                if (h == PD / 64 - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) p_arrive_remote(ro);  // O_t read out (leader's barrier)
                }
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = c8 * 8 + 2 * e;
                        float y0, y1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[col >> 5][col & 31]),
                                                 __uint_as_float(o[col >> 5][(col & 31) + 1])),
                                         inv2),
                                  y0, y1);
                        w4[e] = ppack2<kBF16>(y0, y1);
                    }
                    st_shared_v4(wst + lane * 128 + ((c8 ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = 4 * i + (lane >> 3), ch = lane & 7;
                    const uint4 v4 = ld_shared_v4(wst + rr * 128 + ((ch ^ (rr & 7)) << 4));
                    if (rr < rows_left)
                        *reinterpret_cast<uint4*>(obase + (size_t)rr * (PD * 2) + h * 128 + ch * 16) = v4;
                }
                __syncwarp();
            }
        }
    }

    // every MMA of the leader has completed before this CTA's shared memory and TMEM go
    if (warp == kPMmaWarp && lane == 0) pwait_one(bar.drain, 0, abort_flag, p.status, false);
    tc_fence_before();
    __syncthreads();
    p_cluster_sync();
    if (warp == kPMmaWarp) {
        tc_fence_after();
        p_tmem_dealloc(tmem, 512);
    }
}

template <bool kBF16>
int launch_pair_t(const Problem& pr, const void* q, const void* k, const void* v, void* o, int* status,
                  cudaStream_t stream) {
    static PerDeviceOnce attr_once;
    if (once_per_device(attr_once, [] {
            return cudaFuncSetAttribute(attn_prefill_pair_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kPSmemBytes);
        }) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const int sms = device_sm_count();
    if (sms < 2) return ATTN_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (!make_tensor_map(&tq, q, PD, pr.M, pr.B * pr.Hq, PBM, kBF16) ||
        !make_tensor_map(&tk, k, PD, pr.N, pr.B * pr.Hkv, 64, kBF16) ||
        !make_tensor_map(&tv, v, PD, pr.N, pr.B * pr.Hkv, PBN, kBF16))
        return ATTN_ERR_CUDA;
    PairParams pp;
    pp.o = o;
    pp.lse = pr.lse;
    pp.status = status;
    pp.M = pr.M;
    pp.N = pr.N;
    pp.Hq = pr.Hq;
    pp.Hkv = pr.Hkv;
    pp.G = pr.G;
    pp.causal = pr.causal;
    pp.window = pr.window;
    pp.scale_log2 = pr.scale_log2;
    pp.BH = pr.B * pr.Hq;
    pp.nqb = (pr.M + PRows - 1) / PRows;
    pp.tiles = pp.BH * pp.nqb;
    const int pairs = pp.tiles < sms / 2 ? pp.tiles : sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_prefill_pair_kernel<kBF16>, tq, tk, tv, pp);
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

bool prefill_pair_supported(const Problem& p) {
    return p.D == PD && (int64_t)p.B * p.Hq * ((p.M + PRows - 1) / PRows) < (1LL << 31);
}

int launch_prefill_pair(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                        cudaStream_t stream) {
    if (p.D != PD) return ATTN_ERR_HEADDIM;
    return p.dtype == ATTN_BF16 ? launch_pair_t<true>(p, q, k, v, o, status, stream)
                                : launch_pair_t<false>(p, q, k, v, o, status, stream);
}

}  // namespace attn
