// Prefill forward on the 5th-generation tensor cores (tcgen05 + TMEM), sm_103a.
//
// Persistent kernel: one CTA per SM walks a list of work tiles, each two
// 128-row query tiles (256 rows) of one (batch, head), and streams the
// key/value tiles they may see. Warp roles:
//   warps 0-3  softmax + epilogue for query tile 0 (one TMEM lane = one row = one thread)
//   warps 4-7  softmax + epilogue for query tile 1
//   warp 8     TMA producer: Q of each work tile, then K_j, V_j through a shared-memory ring
//   warp 9     MMA issuer (whole warp, one elected lane issues): S_t = Q_t K_j^T and O_t += P_t V_j
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
// boundary checks are not free). Key tiles that no row of a work tile may see
// are never loaded (causal and window tile skipping).
//
// Work tiles are ordered longest first (causal) and dealt to the CTAs in a
// serpentine order, which balances causal work to about 1 %. Across work
// tiles the K/V ring and every barrier phase carry on: Q of the next tile is
// loaded as soon as the last score product of the current one has read Q, and
// the next tile's first value product into O_t waits only until the epilogue
// of the current tile has pulled O_t out of TMEM, so epilogues overlap MMAs.
// Each query tile's epilogue starts as soon as its own last value product has
// completed (one O-final barrier per tile), about one softmax step before the
// other tile's.
// The epilogue goes through shared memory: each softmax warp writes its 32
// normalized rows of a 64-column half into its own 4 KB area (16-byte chunks in
// a 128-byte swizzle) and copies them out with stores of four whole 128-byte
// row segments per instruction. A row-per-thread global store would touch 32
// rows per instruction and hold up the next tile's TMEM reads; a TMA store of
// the area would queue behind the next tile's Q and K/V loads in the SM's TMA
// unit (measured: about 4,000 cycles at every work-tile transition).
//
// The issuer keeps the tensor pipe fed only if it spends little time per MMA
// and between MMA groups (the pipe queues about one MMA). The whole warp runs
// the issuing loop, so descriptors and TMEM addresses are warp-uniform values,
// and one elected lane issues each instruction; run by one divergent thread,
// the same loop took about 83 cycles per MMA, against 64 of tensor work for a
// 128 x 128 x 16 product, and the kernel 10 % longer. The issuer also makes one
// commit per key tile for the ring (after S_1(j), freeing K_j and V_(j-1)
// together) and tests the readiness of V_j and P_0(j) between the two halves
// of the S_1(j) group, while queued MMAs run, instead of waiting after it.
//
// Rescaling is lazy: a row's reference maximum moves only when the new
// maximum exceeds it by more than 8 (base-2 units), so p = 2^(t - m_ref) <= 256
// and the accumulator is rescaled by alpha = 2^(m_old - m_new) only then. The
// final O / l is the same quotient as with an always-current maximum.
//
// Every wait is bounded (1 s); on expiry the CTA raises an abort flag, sets
// the device status word, drains its in-flight copies and MMAs, frees TMEM
// and exits.
//
// The same kernel takes 8-bit E4M3 inputs (kIn = kInE4M3): both products run
// as kind::f8f6f4 with 32-element K steps, a D = 128 row is one 128-byte
// swizzle chunk, and P is rounded to E4M3, four per TMEM column.
#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "tma_map.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int BM = 128;  // rows per query tile
constexpr int BN = 128;  // keys per key/value tile
constexpr int NQ = 2;    // query tiles per work tile
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint64_t kTimeoutNs = 1000000000ull;
constexpr float kRescaleThreshold = 8.0f;

// Input element kinds: 16-bit (output of the same type) or 8-bit E4M3 (output BF16 or FP16).
constexpr int kInF16 = 0, kInBF16 = 1, kInE4M3 = 2;

template <int D, int EB>  // EB: bytes per input element
struct Cfg {
    static constexpr int kRowBytes = D * EB;
    static constexpr int kChunks = kRowBytes / 128;   // 128-byte swizzle chunks along D
    static constexpr int kChunkElems = 128 / EB;      // elements of D per chunk
    static constexpr int kChunkBytes = BM * 128;      // one chunk of a 128-row tile
    static constexpr int kTileBytes = BM * kRowBytes; // one Q, K or V tile
    static constexpr int kStages = (kRowBytes == 256) ? 4 : 8;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = NQ * kTileBytes;
    // output staging: 4 KB per softmax warp (its 32 rows x 64 columns of 16-bit output)
    static constexpr int kStageOff = kKVOff + kStages * kTileBytes;
    static constexpr int kBarOff = kStageOff + 8 * 4096;
    // q_full, q_free, full[S], empty[S], s_full[2], p_full[2], o_final[2], o_free[2], drain
    static constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 2 + 2 + 1;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
};

// TMEM column of S_t / P_t and of O_t
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }

struct PrefillParams {
    void* o;
    float* lse;  // optional per-row log-sum-exp (natural log)
    int* status;
    int M, N, Hq, Hkv, G;
    int causal, window;
    float scale_log2;  // for 8-bit inputs this includes the Q and K dequantization factors
    float v_scale;     // V dequantization factor (1 for 16-bit inputs), applied with 1 / l
    int BH;     // B * Hq
    int nqb;    // work tiles per head (ceil(M / 256))
    int tiles;  // BH * nqb
    // > 0: walk the heads in groups of this many (every work tile has the same
    // length); 0: all heads' last query blocks first, longest first
    int head_group;
    // failure-path self-test only (-1 otherwise): the softmax warps of query tile 0
    // withhold their P-ready arrival for this score tile (counted over the CTA's walk),
    // so the issuing warp's bounded wait runs out and the whole CTA takes its abort path
    long withhold_p_at;
};

struct Bars {
    uint32_t q_full, q_free, full0, empty0, s0, p0, o_final0, o_free0, drain;
    __device__ uint32_t full(int s) const { return full0 + 8u * s; }
    __device__ uint32_t empty(int s) const { return empty0 + 8u * s; }
    __device__ uint32_t s_full(int t) const { return s0 + 8u * t; }
    __device__ uint32_t p_full(int t) const { return p0 + 8u * t; }
    __device__ uint32_t o_final(int t) const { return o_final0 + 8u * t; }
    __device__ uint32_t o_free(int t) const { return o_free0 + 8u * t; }
};

// Geometry of one work tile: its head, first row and the key tiles it visits.
struct Work {
    int bh, kvh, row0, jt0, n;
};

// w-th work tile of this CTA (serpentine over a longest-first order); false when done.
__device__ __forceinline__ bool work_tile(const PrefillParams& p, int w, Work* t) {
    const int grid = gridDim.x, c = blockIdx.x;
    const int idx = w * grid + ((w & 1) ? grid - 1 - c : c);
    if (idx >= p.tiles) return false;
    int qb;
    if (p.head_group > 0) {
        // equal work tiles: a group of heads at a time, so that the K/V the CTAs
        // running at once read (a few heads' worth) stays in L2
        const int per = p.head_group * p.nqb;
        const int h0 = (idx / per) * p.head_group, j = idx % per;
        const int hn = min(p.head_group, p.BH - h0);
        qb = p.nqb - 1 - j / hn;
        t->bh = h0 + j % hn;
    } else {
        // longest work tiles first over all heads (causal and window tiles differ
        // in length): the last wave holds the shortest ones
        qb = p.nqb - 1 - idx / p.BH;
        t->bh = idx % p.BH;
    }
    const int b = t->bh / p.Hq, h = t->bh % p.Hq;
    t->kvh = b * p.Hkv + h / p.G;
    t->row0 = qb * (NQ * BM);
    const int off = p.N - p.M;  // row i sits at key position i + off
    const int last_row = min(t->row0 + NQ * BM - 1, p.M - 1);
    int klo = 0, khi = p.N, unused = 0;
    key_range(t->row0 + off, p.N, p.causal, p.window, &klo, &unused);
    key_range(last_row + off, p.N, p.causal, p.window, &unused, &khi);
    t->jt0 = klo / BN;
    t->n = (khi > klo) ? (khi + BN - 1) / BN - t->jt0 : 0;
    return true;
}

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

// Warp-uniform readiness test (true only if every lane saw the phase complete).
__device__ __forceinline__ bool test_warp(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_test(bar, parity));
}

// Warp-uniform bounded wait that ignores the abort flag (for the final drain).
__device__ bool wait_warp_final(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        int stop = 0;
        if ((threadIdx.x & 31) == 0 && globaltimer_ns() - t0 > kTimeoutNs) {
            atomicExch(status, 1);
            stop = 1;
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    return kBF16 ? pack_bf16(lo, hi) : pack_f16(lo, hi);
}

// MMA groups issued from precomputed descriptors: the issuing warp must
// keep up with the tensor core (a 128x128 MMA step retires in 64 cycles for
// 16-bit inputs, 32 for 8-bit), so each K step only adds a compile-time offset
// to a 64-bit descriptor. Every K step covers 32 bytes of a row: 16 elements
// of 16 bits or 32 of 8 bits.
template <int D, int EB, class F>
__device__ __forceinline__ void mma_group_s(uint32_t d_tmem, uint64_t a0, uint64_t b0, uint32_t idesc, F&& between) {
#pragma unroll
    for (int kk = 0; kk < D * EB / 32; ++kk) {
        if (kk == D * EB / 64) between();
        const uint64_t off = (uint64_t)((((kk >> 2) * Cfg<D, EB>::kChunkBytes) + (kk & 3) * 32) >> 4);
        if constexpr (EB == 1)
            mma_ss_f8_el(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
        else
            mma_ss_el(d_tmem, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
    }
}
// P from TMEM (8 columns per K step: two 16-bit or four 8-bit values per
// column), V from a shared-memory slot (MN-major: one K step is kKStep key rows)
template <int EB>
__device__ __forceinline__ void mma_group_pv(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, uint32_t idesc,
                                             bool first) {
    constexpr int kStep = 32 / EB;
#pragma unroll
    for (int kk = 0; kk < BN / kStep; ++kk) {
        const uint64_t b = b0 + (uint64_t)((kk * kStep * 128) >> 4);
        if constexpr (EB == 1)
            mma_ts_f8_el(d_tmem, a_tmem + kk * 8, b, idesc, (first && kk == 0) ? 0u : 1u);
        else
            mma_ts_el(d_tmem, a_tmem + kk * 8, b, idesc, (first && kk == 0) ? 0u : 1u);
    }
}

// kBF16: output type (and input type for 16-bit inputs). DO: columns of the
// tensors and the output (D, or 64 for 8-bit inputs run as D = 128: the upper
// 64 columns of every Q, K and V tile read as zeros and are never written out).
template <int D, int kIn, bool kBF16, int DO = D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    constexpr int EB = kIn == kInE4M3 ? 1 : 2;
    using C = Cfg<D, EB>;
    constexpr int kHalf = C::kStages / 2;  // empty barriers: one per pair of slots freed together
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kQOff;
    const uint32_t sKV = sbase + C::kKVOff;
    const uint32_t sStage = sbase + C::kStageOff;
    Bars bar;
    bar.q_full = sbase + C::kBarOff;
    bar.q_free = bar.q_full + 8;
    bar.full0 = bar.q_free + 8;
    bar.empty0 = bar.full0 + 8 * C::kStages;
    bar.s0 = bar.empty0 + 8 * C::kStages;
    bar.p0 = bar.s0 + 16;
    bar.o_final0 = bar.p0 + 16;
    bar.o_free0 = bar.o_final0 + 16;
    bar.drain = bar.o_free0 + 16;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(bar.q_full, 1);
        mbar_init(bar.q_free, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar.full(s), 1);
            mbar_init(bar.empty(s), 1);
        }
        for (int t = 0; t < NQ; ++t) {
            mbar_init(bar.s_full(t), 1);
            mbar_init(bar.p_full(t), 4);  // one arrival per softmax warp
            mbar_init(bar.o_free(t), 4);
        }
        mbar_init(bar.o_final(0), 1);
        mbar_init(bar.o_final(1), 1);
        mbar_init(bar.drain, 1);
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
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            int u = 0, tc = 0;  // ring position and work tiles with keys, across the whole walk
            int q_issued = 0;   // Q loads issued
            bool ok = true;
            Work wk;
            for (int w = 0; ok && work_tile(p, w, &wk); ++w) {
                if (wk.n == 0) continue;
                // Q of this tile may overwrite Q of the previous one once its last score product read it
                if (tc > 0 && !(ok = wait_one(bar.q_free, (tc - 1) & 1, abort_flag, p.status))) break;
                mbar_arrive_expect_tx(bar.q_full, NQ * C::kTileBytes);
                for (int t = 0; t < NQ; ++t)
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sQ + t * C::kTileBytes + c * C::kChunkBytes, &tmQ, c * C::kChunkElems, wk.row0 + t * BM,
                                    wk.bh, bar.q_full);
                ++q_issued;
                // K_j and V_j alternate through the ring in the order the MMA uses them.
                // One commit after S_1(J) frees K_J and V_(J-1) (empty barrier J % kHalf, phase
                // J / kHalf); K_J reuses K_(J-kHalf)'s slot and V_J reuses V_(J-kHalf)'s.
                for (int x = 0; x < 2 * wk.n; ++x, ++u) {
                    const int s = u % C::kStages;
                    const int J = u >> 1;
                    const int Jf = (u & 1) ? J - kHalf + 1 : J - kHalf;  // the step whose commit frees this slot
                    if (u >= C::kStages &&
                        !(ok = wait_one(bar.empty(Jf % kHalf), (Jf / kHalf) & 1, abort_flag, p.status)))
                        break;
                    mbar_arrive_expect_tx(bar.full(s), C::kTileBytes);
                    const CUtensorMap* tm = (x & 1) ? &tmV : &tmK;
                    const int key0 = (wk.jt0 + x / 2) * BN;
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(sKV + s * C::kTileBytes + c * C::kChunkBytes, tm, c * C::kChunkElems, key0, wk.kvh,
                                    bar.full(s));
                }
                ++tc;
            }
            // every issued copy must land before the CTA may exit
            if (q_issued > 0) wait_one(bar.q_full, (q_issued - 1) & 1, abort_flag, p.status, false);
            for (int x = max(0, u - C::kStages); x < u; ++x)
                wait_one(bar.full(x % C::kStages), (x / C::kStages) & 1, abort_flag, p.status, false);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        // The whole warp runs the loop (operands stay warp-uniform); one elected lane
        // issues each MMA and commit.
        {
            constexpr uint32_t idS = EB == 1 ? idesc_e4m3(BM, BN, false) : idesc_f16(kBF16, BM, BN, false);
            constexpr uint32_t idPV = EB == 1 ? idesc_e4m3(BM, D, true) : idesc_f16(kBF16, BM, D, true);
            int u = 0, tc = 0;
            int ps[NQ] = {0, 0};  // P tiles consumed per query tile, across the walk
            bool ok = true;
            // descriptors: Q_0, Q_1, and ring slot 0 (K-major for K, MN-major for V);
            // slot s adds s * kTileBytes to the 14-bit address field
            const uint64_t dq0 = sw128_desc(sQ, 16, 1024);
            const uint64_t dq1 = sw128_desc(sQ + C::kTileBytes, 16, 1024);
            const uint64_t dk = sw128_desc(sKV, 16, 1024);
            const uint64_t dv = sw128_desc(sKV, C::kChunkBytes, 1024);
            constexpr uint64_t kSlotStep = (uint64_t)(C::kTileBytes >> 4);
            auto issue_s = [&](int t, int slot) {
                mma_group_s<D, EB>(tmem + col_s(t), t ? dq1 : dq0, dk + (uint64_t)slot * kSlotStep, idS, [] {});
            };
            // O_t += P_t V; the first product of a tile overwrites O_t, after the
            // previous tile's epilogue has read it out
            bool p_ready = false;  // P_0's phase was seen complete in the middle of the S_1 group
            auto issue_pv = [&](int t, int slot, bool first) {
                if (!(t == 0 && p_ready) && !wait_warp(bar.p_full(t), ps[t] & 1, abort_flag, p.status)) return false;
                ++ps[t];
                if (first && tc > 0 && !wait_warp(bar.o_free(t), (tc - 1) & 1, abort_flag, p.status)) return false;
                tc_fence_after();
                mma_group_pv<EB>(tmem + col_o(t), tmem + col_s(t), dv + (uint64_t)slot * kSlotStep, idPV, first);
                return true;
            };
            Work wk;
            for (int w = 0; ok && work_tile(p, w, &wk); ++w) {
                const int n = wk.n;
                if (n == 0) continue;
                if (!(ok = wait_warp(bar.q_full, tc & 1, abort_flag, p.status))) break;
                tc_fence_after();
                int slot_v_prev = 0;
                for (int jj = 0; jj < n; ++jj) {
                    const int uk = u++, sk = uk % C::kStages;
                    const int uv = u++, sv = uv % C::kStages;
                    if (!(ok = wait_warp(bar.full(sk), (uk / C::kStages) & 1, abort_flag, p.status))) break;
                    tc_fence_after();
                    issue_s(0, sk);
                    mma_commit_el(bar.s_full(0));
                    if (jj > 0) {
                        if (!(ok = issue_pv(1, slot_v_prev, jj - 1 == 0))) break;
                    }
                    // S_1, with the readiness of V_j and P_0 tested between its halves (a test
                    // there overlaps the MMAs already queued; a wait after the group does not)
                    bool v_ready = false;
                    p_ready = false;
                    mma_group_s<D, EB>(tmem + col_s(1), dq1, dk + (uint64_t)sk * kSlotStep, idS, [&] {
                        v_ready = test_warp(bar.full(sv), (uv / C::kStages) & 1);
                        p_ready = test_warp(bar.p_full(0), ps[0] & 1);
                    });
                    mma_commit_el(bar.s_full(1));
                    if (jj == n - 1) mma_commit_el(bar.q_free);  // Q is read for the last time
                    mma_commit_el(bar.empty((uk >> 1) % kHalf));  // K_j and V_(j-1) are read
                    if (!v_ready && !(ok = wait_warp(bar.full(sv), (uv / C::kStages) & 1, abort_flag, p.status))) break;
                    if (!(ok = issue_pv(0, sv, jj == 0))) break;
                    if (jj == n - 1) mma_commit_el(bar.o_final(0));  // O_0 of this tile is final
                    slot_v_prev = sv;
                }
                if (!ok) break;
                if (!(ok = issue_pv(1, slot_v_prev, n - 1 == 0))) break;
                mma_commit_el(bar.o_final(1));  // O_1 of this tile is final
                ++tc;
            }
            // all MMAs done before TMEM and shared memory are released
            mma_commit_el(bar.drain);
            wait_warp_final(bar.drain, 0, p.status);
        }
        __syncwarp();
    } else {
        // ---------------- softmax warps ----------------
        const int t = warp >> 2;  // query tile
        const int wq = warp & 3;  // TMEM lane quarter
        const int r_in_tile = wq * 32 + lane;
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const uint32_t tS = tmem + lane_base + col_s(t);
        const uint32_t tO = tmem + lane_base + col_o(t);
        const float c = p.scale_log2;
        const float masked_s = c >= 0.f ? -INFINITY : INFINITY;  // scores that give t = -inf
        const int off = p.N - p.M;
        int g = 0, tc = 0;  // score tiles and work tiles with keys, across the walk
        bool ok = true;
        Work wk;
        for (int w = 0; ok && work_tile(p, w, &wk); ++w) {
            const int row = wk.row0 + t * BM + r_in_tile;
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) + ((size_t)wk.bh * p.M + row) * DO;
            if (wk.n == 0) {  // no row of this tile sees any key: output 0
                if (row < p.M) {
                    if (p.lse) p.lse[(size_t)wk.bh * p.M + row] = -INFINITY;
                    uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
                    for (int v4 = 0; v4 < DO / 8; ++v4) dst[v4] = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            const int pos = row + off;
            const int tile_first_pos = wk.row0 + t * BM + off;
            const int tile_last_pos = tile_first_pos + BM - 1;
            float m_ref = -INFINITY;  // reference maximum (base-2 scaled units)
            float l = 0.f;
            for (int jj = 0; jj < wk.n; ++jj, ++g) {
                const int key0 = (wk.jt0 + jj) * BN;
                if (!(ok = wait_warp(bar.s_full(t), g & 1, abort_flag, p.status))) break;
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
                    const int vlo = lo - key0, vhi = hi - key0;  // this row's visible columns of the tile
                    if (p.window > 0) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (q4 * 32 + e < vlo || q4 * 32 + e >= vhi) s[q4][e] = __float_as_uint(masked_s);
                    } else {  // no window: vlo <= 0, only the end of the range cuts
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (q4 * 32 + e >= vhi) s[q4][e] = __float_as_uint(masked_s);
                    }
                }
                // row maximum (minimum for a negative scale) with three-input operations
                float mx;
                {
#define SV(i) __uint_as_float(s[(i) >> 5][(i) & 31])
                    // eight chains over 16 columns each (depth 8), then a two-level tree
                    float a[8];
                    if (c >= 0.f) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            a[k] = max3f(SV(16 * k), SV(16 * k + 1), SV(16 * k + 2));
#pragma unroll
                            for (int e = 3; e < 15; e += 2) a[k] = max3f(a[k], SV(16 * k + e), SV(16 * k + e + 1));
                            a[k] = fmaxf(a[k], SV(16 * k + 15));
                        }
                        mx = max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            a[k] = min3f(SV(16 * k), SV(16 * k + 1), SV(16 * k + 2));
#pragma unroll
                            for (int e = 3; e < 15; e += 2) a[k] = min3f(a[k], SV(16 * k + e), SV(16 * k + e + 1));
                            a[k] = fminf(a[k], SV(16 * k + 15));
                        }
                        mx = min3f(min3f(a[0], a[1], a[2]), min3f(a[3], a[4], a[5]), fminf(a[6], a[7]));
                    }
#undef SV
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
                // p = 2^(s c - m_use) for pairs of keys (packed FMA), summed into l
                // in two packed chains, rounded to the P type and written over S
                const uint64_t c2 = f2_pack(c, c), nm2 = f2_pack(-m_use, -m_use);
                uint64_t lsum[2] = {0ull, 0ull};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    if constexpr (EB == 2) {
                        uint32_t packed[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[q4][2 * e]), __uint_as_float(s[q4][2 * e + 1])),
                                             c2, nm2),
                                      x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            lsum[e & 1] = f2_add(lsum[e & 1], f2_pack(p0, p1));
                            packed[e] = pack2<kBF16>(p0, p1);
                        }
                        tmem_st_x16(tS + q4 * 16, packed);  // P overwrites the first 64 columns of S
                    } else {
                        // P rounded to E4M3 for the value product (p <= 256 < 448); l
                        // sums the unrounded FP32 values
                        uint32_t packed[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float pv[4];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int e2 = 2 * e + h;
                                float x0, x1;
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(s[q4][2 * e2]),
                                                         __uint_as_float(s[q4][2 * e2 + 1])),
                                                 c2, nm2),
                                          x0, x1);
                                pv[2 * h] = ex2(x0);
                                pv[2 * h + 1] = ex2(x1);
                                lsum[h] = f2_add(lsum[h], f2_pack(pv[2 * h], pv[2 * h + 1]));
                            }
                            packed[e] = pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
                        }
                        tmem_st_x8(tS + q4 * 8, packed);  // P overwrites the first 32 columns of S
                    }
                }
                {
                    float l0, l1, l2, l3;
                    f2_unpack(lsum[0], l0, l1);
                    f2_unpack(lsum[1], l2, l3);
                    l += (l0 + l1) + (l2 + l3);
                }
                // rescale the accumulator (the value product of the previous key tile
                // has completed: its commit preceded this tile's score commit)
                if (__any_sync(0xffffffffu, need) && jj > 0) {
#pragma unroll
                    for (int ch = 0; ch < D / 32; ++ch) {
                        uint32_t o[32];
                        tmem_ld_x32(tO + ch * 32, o);
                        tmem_wait_ld_x32(o);
                        const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            float y0, y1;
                            f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), a2), y0,
                                      y1);
                            o[2 * e] = __float_as_uint(y0);
                            o[2 * e + 1] = __float_as_uint(y1);
                        }
                        tmem_st_x32(tO + ch * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();  // the warp's TMEM stores are ordered before lane 0's arrival
                if (lane == 0 && !(t == 0 && g == p.withhold_p_at)) mbar_arrive(bar.p_full(t));
            }
            if (!ok) break;

            // ---------------- epilogue: O / l, one cast, rows < M ----------------
            // Per 64-column half: each warp writes its 32 rows, normalized and cast,
            // into its own 4 KB staging area (16-byte chunks in a 128-byte swizzle, so
            // neither the writes nor the reads conflict), then copies them out with
            // 16-byte stores of four whole 128-byte row segments per instruction
            // (a row-per-thread store would touch 32 rows per instruction).
            if (!(ok = wait_warp(bar.o_final(t), tc & 1, abort_flag, p.status))) break;
            ++tc;
            tc_fence_after();
            const float inv = l > 0.f ? p.v_scale / l : 0.f;  // no visible key: output 0
            // log sum_j e^(scale s_j) = ln 2 * (m_ref + log2 l) (p was taken against m_ref)
            if (p.lse && row < p.M)
                p.lse[(size_t)wk.bh * p.M + row] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
            const uint32_t wst = sStage + (t * 4 + wq) * 4096;  // this warp's staging area
            const uint64_t inv2 = f2_pack(inv, inv);
            char* obase = reinterpret_cast<char*>(p.o) + ((size_t)wk.bh * p.M + wk.row0 + t * BM + wq * 32) * (DO * 2);
            const int rows_left = p.M - (wk.row0 + t * BM + wq * 32);  // rows of this warp below M
#pragma unroll
            for (int h = 0; h < DO / 64; ++h) {
                uint32_t o[2][32];
                tmem_ld_x32(tO + h * 64, o[0]);
                tmem_ld_x32(tO + h * 64 + 32, o[1]);
                tmem_wait_ld_x32(o[0]);
                reg_after_x32(o[1]);
                if (h == DO / 64 - 1) {
                    // O_t is read out: it may take the next tile's first value product
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar.o_free(t));
                }
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {  // 16-byte chunk c8: columns 8 c8 .. 8 c8 + 7 of the half
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int col = c8 * 8 + 2 * e;
                        float y0, y1;
                        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[col >> 5][col & 31]),
                                                 __uint_as_float(o[col >> 5][(col & 31) + 1])),
                                         inv2),
                                  y0, y1);
                        w4[e] = pack2<kBF16>(y0, y1);
                    }
                    st_shared_v4(wst + lane * 128 + ((c8 ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 8; ++i) {  // rows 4 i .. 4 i + 3 of the warp, one 16-byte chunk per lane
                    const int rr = 4 * i + (lane >> 3), ch = lane & 7;
                    const uint4 v4 = ld_shared_v4(wst + rr * 128 + ((ch ^ (rr & 7)) << 4));
                    if (rr < rows_left)
                        *reinterpret_cast<uint4*>(obase + (size_t)rr * (DO * 2) + h * 128 + ch * 16) = v4;
                }
                __syncwarp();  // the area is read before the next half overwrites it
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

template <int D, int kIn, bool kBF16, int DO = D>
int launch_t(const Problem& pr, const void* q, const void* k, const void* v, void* o, int* status, float v_scale,
             cudaStream_t stream, long withhold_p_at = -1) {
    constexpr int EB = kIn == kInE4M3 ? 1 : 2;
    using C = Cfg<D, EB>;
    static PerDeviceOnce attr_once;
    if (once_per_device(attr_once, [] {
            return cudaFuncSetAttribute(attn_prefill_kernel<D, kIn, kBF16, DO>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        }) != cudaSuccess)
        return ATTN_ERR_CUDA;
    const int sms = device_sm_count();
    if (sms <= 0) return ATTN_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (!make_tensor_map(&tq, q, DO, pr.M, pr.B * pr.Hq, BM, kBF16, EB) ||
        !make_tensor_map(&tk, k, DO, pr.N, pr.B * pr.Hkv, BN, kBF16, EB) ||
        !make_tensor_map(&tv, v, DO, pr.N, pr.B * pr.Hkv, BN, kBF16, EB))
        return ATTN_ERR_CUDA;
    PrefillParams pp;
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
    pp.v_scale = v_scale;
    pp.BH = pr.B * pr.Hq;
    pp.nqb = (pr.M + NQ * BM - 1) / (NQ * BM);
    pp.tiles = pp.BH * pp.nqb;
    pp.withhold_p_at = withhold_p_at;
    const int grid = pp.tiles < sms ? pp.tiles : sms;
    // Work tiles of equal length (no causal mask, no window) over at least four
    // waves: heads in groups of about one wave's worth of tiles (measured: the
    // D = 128 noncausal 4096 workload 3.5 % faster; with 1.7 waves, or tiles of
    // different lengths, the all-heads longest-first order is faster).
    pp.head_group = (!pr.causal && pr.window <= 0 && pp.tiles >= 4 * grid) ? (grid + pp.nqb - 1) / pp.nqb : 0;
    attn_prefill_kernel<D, kIn, kBF16, DO><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, pp);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

bool prefill_supported(const Problem& p) {
    return (p.D == 64 || p.D == 128) && (int64_t)p.B * p.Hq * ((p.M + NQ * BM - 1) / (NQ * BM)) < (1LL << 31);
}

int launch_prefill(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                   cudaStream_t stream) {
    const bool bf16 = p.dtype == ATTN_BF16;
    if (p.D == 128) return bf16 ? launch_t<128, kInBF16, true>(p, q, k, v, o, status, 1.f, stream)
                                : launch_t<128, kInF16, false>(p, q, k, v, o, status, 1.f, stream);
    if (p.D == 64) return bf16 ? launch_t<64, kInBF16, true>(p, q, k, v, o, status, 1.f, stream)
                               : launch_t<64, kInF16, false>(p, q, k, v, o, status, 1.f, stream);
    return ATTN_ERR_HEADDIM;
}

int launch_prefill_withheld(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                            long withhold_p_at, cudaStream_t stream) {
    if (p.D != 128) return ATTN_ERR_HEADDIM;
    return p.dtype == ATTN_BF16
               ? launch_t<128, kInBF16, true>(p, q, k, v, o, status, 1.f, stream, withhold_p_at)
               : launch_t<128, kInF16, false>(p, q, k, v, o, status, 1.f, stream, withhold_p_at);
}

int launch_prefill_e4m3(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                        float v_scale, cudaStream_t stream) {
    if (p.D == 128)
        return p.dtype == ATTN_BF16 ? launch_t<128, kInE4M3, true>(p, q, k, v, o, status, v_scale, stream)
                                    : launch_t<128, kInE4M3, false>(p, q, k, v, o, status, v_scale, stream);
    // D = 64: the 128-column kernel on 64-byte rows read through 128-byte boxes
    // (columns 64..127 read as zeros), writing 64 output columns
    if (p.D == 64)
        return p.dtype == ATTN_BF16 ? launch_t<128, kInE4M3, true, 64>(p, q, k, v, o, status, v_scale, stream)
                                    : launch_t<128, kInE4M3, false, 64>(p, q, k, v, o, status, v_scale, stream);
    return ATTN_ERR_HEADDIM;
}

}  // namespace attn
