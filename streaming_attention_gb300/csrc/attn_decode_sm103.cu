// Split-KV decode on the tcgen05 tensor cores (sm_103a), D = 128 (and D = 64 for
// 16-bit inputs, read as D = 128 with the upper 64 columns zero).
//
// Decode has few query rows per KV head: the R = (Hq/Hkv) * M rows that share
// one KV head (GQA grouping) are processed together, padded to 16; more than 16
// are cut into blocks of 16 rows, one CTA each along the grid's z (each streams
// the split's K/V tiles; the blocks of one split run side by side, so their
// re-reads of the same tiles mostly hit L2). The score
// tile is computed transposed, S^T[128 keys x 16 rows] = K_tile Q^T, so the
// 128 keys fill the MMA's M dimension instead of 112 padded query rows; then
// O^T[128 dims x 16 rows] += V_tile^T P^T. One thread owns one key for the
// softmax (TMEM lane = key) and one head dimension for the accumulator (TMEM
// lane = d). The row maximum of a tile is reduced across the 128 threads with
// warp shuffles and a shared-memory exchange; row sums stay per-thread until
// the end.
//
// Each CTA streams one split (a run of 128-key tiles) of one KV head through a
// TMA ring (3 slots of 16-bit tiles, 6 of 8-bit tiles), K and V tiles in the
// order the MMAs consume them (for the 8-bit contiguous cache in rounds of two
// tiles, so the softmax's cross-warp maximum exchange and P handshake come once
// per 256 keys), and forms the split's unnormalized summary
// (m, l, acc) for its rows. The summaries are combined with the common-maximum
// rule ("Compare reasoning after your own attempt", central-idea table, A1 and
// A2 rows): when a KV head has at most 8 splits they form one thread-block
// cluster and merge through distributed shared memory, each CTA writing some
// of the output rows; otherwise they go to the workspace for the merge kernel.
// Masks, ghost rows, lazy rescale and bounded waits follow the prefill kernel.
#include <mutex>

#include "attn_internal.h"
#include "sm100_ptx.cuh"
#include "tma_map.h"

namespace attn {
namespace {

using namespace ptx;

constexpr int DBN = 128;  // keys per tile (MMA M of the score product)
constexpr int DNR = 16;   // grouped rows, padded (MMA N)
constexpr int DD = 128;   // head dimension (MMA M of the value product)
constexpr int kDecThreads = 192;  // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int kDecLoadWarp = 4, kDecMmaWarp = 5;
constexpr uint64_t kDecTimeoutNs = 1000000000ull;
constexpr float kDecRescale = 8.0f;

constexpr int kChunkBytes = DBN * 128;  // one 128-byte column chunk of a 128-row tile
constexpr int kQChunk = DNR * 128;      // one 128-byte column chunk of the 16-row Q or P^T tile

// Shared-memory plan for EB-byte inputs (2: BF16/FP16, 1: E4M3). The ring keeps
// about 96 KB of K/V in flight per CTA either way (3 slots of 32 KB, 6 of 16 KB),
// and two CTAs share an SM. (Three 8-bit CTAs per SM with 3 slots each, and
// so more splits, measured slower: the extra merge work outweighed the gain.)
template <int EB>
struct DCfg {
    static constexpr int kSlots = EB == 1 ? 6 : 3;
    static constexpr int kTileBytes = DBN * DD * EB;  // K or V tile
    static constexpr int kChunks = DD * EB / 128;     // column chunks of a row
    static constexpr int kChunkElems = 128 / EB;      // elements of D per chunk
    static constexpr int kQBytes = DNR * DD * EB;
    static constexpr int kPBytes = DNR * DBN * EB;    // one P^T buffer
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kQBytes;     // two P^T buffers
    static constexpr int kOffRing = 12288;            // 1024-aligned
    static constexpr int kOffBar = kOffRing + kSlots * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kSlots + 2 + 2 + 2 + 1 + 2 + 1;
    static constexpr int kOffRed = kOffBar + 8 * kNumBars;  // float [2][4][16] tile maxima
    static constexpr int kOffLRed = kOffRed + 2 * 4 * DNR * 4;  // float [4][16] row sums
    static constexpr int kOffMisc = kOffLRed + 4 * DNR * 4;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
};

// TMEM columns: S^T buffers at 0 and 16, O^T at 32
constexpr uint32_t kTmemCols = 64;
__host__ __device__ constexpr uint32_t dcol_s(int b) { return b ? 16u : 0u; }
constexpr uint32_t kColOT = 32;

struct DecodeParams {
    float* ws_m;
    float* ws_l;
    float* ws_acc;
    int* status;
    int Hq, Hkv, M, N, G;
    int R;  // grouped query rows per KV head (G * M); CTA z takes rows [16 z, 16 z + 16) of them
    int D;  // head dimension of the tensors: 128, or 64 (16-bit), whose upper 64 columns read as zeros
    int causal, window;
    float scale_log2;
    int klo, khi, kbase, chunk, S;
    // paged KV cache: K/V pools [pages][Hkv][page_size][D]; sequence b's key j is
    // row j % page_size of page block_table[b][j / page_size]; b holds seq_lens[b] keys
    const int* block_table;
    const int* seq_lens;
    int page_size, max_pages, max_len;
    int oob_z;  // a pool coordinate past its last (page, head): TMA reads zeros there
    // cluster merge (the S <= 8 splits of a group are one thread-block cluster):
    // the CTAs combine the summaries through distributed shared memory, each
    // writing some of the output rows and their log-sum-exp, so no merge kernel runs
    int cluster;
    void* o;
    float* lse;
    int out_dtype;
    float out_scale;
};

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The closing barrier orders nothing in memory (the remote reads it protects have
// returned their values): a relaxed arrival does not wait for this CTA's global
// stores to complete, as a release would.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// shared-memory address of the same variable in cluster CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Keys of one CTA's sequence: its length and the union [klo, khi) of the
// ranges its M query rows may see; splits start at kbase (a tile boundary).
struct SeqRange {
    int N, klo, khi, kbase;
};

__device__ bool dwait_one(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status,
                          bool abortable = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abortable && *abort_flag) return false;
        if (globaltimer_ns() - t0 > kDecTimeoutNs) {
            *abort_flag = 1u;
            atomicExch(status, 1);
            return false;
        }
    }
}

__device__ bool dwait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag, int* status) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        int stop = 0;
        if (lane == 0) {
            if (*abort_flag) {
                stop = 1;
            } else if (globaltimer_ns() - t0 > kDecTimeoutNs) {
                *abort_flag = 1u;
                atomicExch(status, 1);
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

// Warp-uniform bounded wait that ignores the abort flag (for the final drain).
__device__ bool dwait_warp_final(uint32_t bar, uint32_t parity, int* status) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        int stop = 0;
        if ((threadIdx.x & 31) == 0 && globaltimer_ns() - t0 > kDecTimeoutNs) {
            atomicExch(status, 1);
            stop = 1;
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

// Sequence position u of the ring -> (is V, tile index): K_0, K_1, V_0, K_2, V_1, ..., K_{T-1}, V_{T-2}, V_{T-1}
__device__ __forceinline__ void ring_item(int u, int T, bool* is_v, int* tile) {
    if (u == 2 * T - 1) {
        *is_v = true;
        *tile = T - 1;
    } else if (u == 0) {
        *is_v = false;
        *tile = 0;
    } else if (u & 1) {
        *is_v = false;
        *tile = (u + 1) / 2;
    } else {
        *is_v = true;
        *tile = (u - 2) / 2;
    }
}
// The same for two-tile rounds (8-bit contiguous decode): K_0, K_1, then per round
// i >= 1 K_2i, K_2i+1, V_2i-2, V_2i-1, then the last round's V tiles; the last
// round holds one tile when T is odd.
__device__ __forceinline__ void ring_item2(int u, int T, bool* is_v, int* tile) {
    const int R = (T + 1) / 2;
    if (u < min(2, T)) {
        *is_v = false;
        *tile = u;
        return;
    }
    if (R >= 2) {
        const int full_end = 2 + 4 * (R - 2);  // end of the full rounds 1 .. R-2
        const int nk_last = min(2, T - 2 * (R - 1));
        const int body_end = full_end + nk_last + 2;
        if (u < full_end) {
            const int i = 1 + (u - 2) / 4, o = (u - 2) % 4;
            *is_v = o >= 2;
            *tile = o < 2 ? 2 * i + o : 2 * (i - 1) + (o - 2);
            return;
        }
        if (u < body_end) {
            const int o = u - full_end;
            *is_v = o >= nk_last;
            *tile = o < nk_last ? 2 * (R - 1) + o : 2 * (R - 2) + (o - nk_last);
            return;
        }
        *is_v = true;
        *tile = 2 * (R - 1) + (u - body_end);
        return;
    }
    *is_v = true;
    *tile = u - min(2, T);
}
__device__ __forceinline__ int ring_pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int ring_pos_v(int j, int T) { return j == T - 1 ? 2 * T - 1 : 2 * j + 2; }

// EB: bytes per input element (2: BF16 or FP16 by kBF16; 1: E4M3, both products
// kind::f8f6f4 and P^T rounded to E4M3).
// RP: grouped rows handled by the softmax (R <= RP <= 16); the MMA always uses N = 16.
// kPaged: K/V come from a paged pool through a block table, with a length per sequence.
template <int EB, bool kBF16, int RP, bool kPaged>
__global__ void __launch_bounds__(kDecThreads)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
    using C = DCfg<EB>;
    constexpr int kSlots = C::kSlots;
    constexpr int kTileBytes = C::kTileBytes;
    // 8-bit contiguous decode: two key tiles per softmax round, so the cross-warp
    // maximum exchange and the P handshake happen once per 256 keys
    constexpr bool kR2 = EB == 1 && !kPaged;
    constexpr int kNP = kR2 ? 4 : 2;                  // S^T and P^T buffers
    constexpr uint32_t kCols = kR2 ? 128u : kTmemCols;
    constexpr uint32_t kColO = kR2 ? 64u : kColOT;
    static_assert(C::kOffP + kNP * C::kPBytes <= C::kOffRing, "P^T buffers overlap the ring");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::kOffQ, sP = sbase + C::kOffP, sRing = sbase + C::kOffRing;
    const uint32_t bar_q = sbase + C::kOffBar;
    const uint32_t bar_full0 = bar_q + 8, bar_empty0 = bar_full0 + 8 * kSlots;
    // one P-ready barrier per P^T buffer: the MMA issues S_{j+1} before PV_j, so the
    // softmax may finish tile j+1 before the MMA observes tile j; per-buffer phases
    // cannot run two ahead (S_{j+2} is issued only after PV_j)
    const uint32_t bar_s0 = bar_empty0 + 8 * kSlots, bar_p0 = bar_s0 + 16, bar_free0 = bar_p0 + 16;
    const uint32_t bar_o = bar_free0 + 16;
    const uint32_t bar_red0 = bar_o + 8, bar_lred = bar_red0 + 16;  // shared-memory exchanges of the softmax
    float* red = reinterpret_cast<float*>(smem + C::kOffRed);
    // cluster mode: this split's summary [R][D] acc, then [R] m, [R] l, in the ring once it is idle
    float* part = reinterpret_cast<float*>(smem + C::kOffRing);
    float* lred = reinterpret_cast<float*>(smem + C::kOffLRed);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int grp = blockIdx.y;  // b * Hkv + g
    const int b = grp / p.Hkv, g = grp % p.Hkv;
    const int Dh = EB == 1 ? DD : p.D;  // head dimension of the tensors (8-bit inputs: 128)
    const int rblk = blockIdx.z;  // block of 16 of the group's grouped rows
    const int R = min(DNR, p.R - rblk * DNR);  // rows of this CTA
    const int row_base = (b * p.Hq + g * p.G) * p.M + rblk * DNR;  // first global row of this CTA

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar_full0 + 8 * s, 1);
            mbar_init(bar_empty0 + 8 * s, 1);
        }
        mbar_init(bar_s0, 1);
        mbar_init(bar_s0 + 8, 1);
        mbar_init(bar_p0, 4);  // one arrival per softmax warp
        mbar_init(bar_p0 + 8, 4);
        mbar_init(bar_free0, 1);
        mbar_init(bar_free0 + 8, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_red0, 4);
        mbar_init(bar_red0 + 8, 4);
        mbar_init(bar_lred, 4);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    // P^T buffers start at zero (rows >= R are never written afterwards)
    for (int x = threadIdx.x; x < kNP * C::kPBytes / 16; x += blockDim.x)
        reinterpret_cast<uint4*>(smem + C::kOffP)[x] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == kDecMmaWarp) {
        tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Let the merge grid launch now: its CTAs wait in griddepcontrol.wait, which
    // returns only after this whole grid has finished and its writes are visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // This grid is itself launched programmatically, so the kernel before it in
    // the stream (which may have written Q, K or V, or still read the workspace)
    // can still be running: the setup above touched no global memory; wait here.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    SeqRange sq{p.N, p.klo, p.khi, p.kbase};
    if constexpr (kPaged) {
        // lengths are clamped to what the block table and the split plan cover
        sq.N = min(max(__ldg(p.seq_lens + b), 0), p.max_len);
        int lo0, hi0, lo1, hi1;
        key_range(sq.N - p.M, sq.N, p.causal, p.window, &lo0, &hi0);
        key_range(sq.N - 1, sq.N, p.causal, p.window, &lo1, &hi1);
        sq.klo = lo0;
        sq.khi = max(hi1, lo0);
        sq.kbase = (lo0 / DBN) * DBN;
    }
    const int k0 = sq.kbase + split * p.chunk;  // tile-aligned start of this split
    const int kend = min(k0 + p.chunk, sq.khi);
    const int T = kend > max(k0, sq.klo) ? (kend - k0 + DBN - 1) / DBN : 0;

    if (warp == kDecLoadWarp) {
        if (!kPaged && lane == 0 && T > 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            mbar_arrive_expect_tx(bar_q, C::kQBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_3d(sQ + c * kQChunk, &tmQ, c * C::kChunkElems, row_base, 0, bar_q);
            int issued = 0;
            for (int u = 0; u < 2 * T; ++u) {
                const int s = u % kSlots;
                if (u >= kSlots && !dwait_one(bar_empty0 + 8 * s, ((u / kSlots) - 1) & 1, abort_flag, p.status))
                    break;
                bool is_v;
                int tile;
                if constexpr (kR2)
                    ring_item2(u, T, &is_v, &tile);
                else
                    ring_item(u, T, &is_v, &tile);
                mbar_arrive_expect_tx(bar_full0 + 8 * s, kTileBytes);
                const CUtensorMap* tm = is_v ? &tmV : &tmK;
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sRing + s * kTileBytes + c * kChunkBytes, tm, c * C::kChunkElems, k0 + tile * DBN,
                                grp, bar_full0 + 8 * s);
                issued = u + 1;
            }
            dwait_one(bar_q, 0, abort_flag, p.status, false);
            for (int u = max(0, issued - kSlots); u < issued; ++u)
                dwait_one(bar_full0 + 8 * (u % kSlots), (u / kSlots) & 1, abort_flag, p.status, false);
        } else if (kPaged && T > 0) {
            // The whole warp: lane i < nsub copies the i-th page-sized piece of
            // each tile (one box per page, or per 128 rows of a larger page), so
            // the small boxes of small pages are issued in parallel. A lane
            // loads its page number one K tile ahead and keeps it for the V
            // tile (3 ring positions later). Keys past the sequence and bad
            // page numbers read a coordinate outside the pool: TMA fills zeros.
            if (lane == 0) {
                prefetch_tmap(&tmQ);
                prefetch_tmap(&tmK);
                prefetch_tmap(&tmV);
                mbar_arrive_expect_tx(bar_q, C::kQBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_3d(sQ + c * kQChunk, &tmQ, c * C::kChunkElems, row_base, 0, bar_q);
            }
            const int sub = min(p.page_size, DBN), nsub = DBN / sub;
            const int npages = p.oob_z / p.Hkv;
            auto page_of = [&](int tile) {
                const int key = k0 + tile * DBN + lane * sub;
                return (lane < nsub && key < sq.N)
                           ? __ldg(p.block_table + (size_t)b * p.max_pages + key / p.page_size)
                           : -1;
            };
            int pf = page_of(0), e0 = -1, e1 = -1;
            int issued = 0;
            for (int u = 0; u < 2 * T; ++u) {
                const int s = u % kSlots;
                int ok = 1;
                if (u >= kSlots && lane == 0)
                    ok = dwait_one(bar_empty0 + 8 * s, ((u / kSlots) - 1) & 1, abort_flag, p.status) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                bool is_v;
                int tile;
                ring_item(u, T, &is_v, &tile);
                if (!is_v) {
                    if (tile & 1)
                        e1 = pf;
                    else
                        e0 = pf;
                    if (tile + 1 < T) pf = page_of(tile + 1);
                }
                const int page = (tile & 1) ? e1 : e0;
                if (lane == 0) mbar_arrive_expect_tx(bar_full0 + 8 * s, kTileBytes);
                __syncwarp();
                if (lane < nsub) {
                    const CUtensorMap* tm = is_v ? &tmV : &tmK;
                    const int key = k0 + tile * DBN + lane * sub;
                    const bool in = key < sq.N && page >= 0 && page < npages;
                    const int y = in ? key % p.page_size : 0;
                    const int z = in ? page * p.Hkv + g : p.oob_z;
                    const uint32_t dst = sRing + s * kTileBytes + lane * sub * 128;
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_3d(dst + c * kChunkBytes, tm, c * C::kChunkElems, y, z, bar_full0 + 8 * s);
                }
                issued = u + 1;
            }
            if (lane == 0) {
                dwait_one(bar_q, 0, abort_flag, p.status, false);
                for (int u = max(0, issued - kSlots); u < issued; ++u)
                    dwait_one(bar_full0 + 8 * (u % kSlots), (u / kSlots) & 1, abort_flag, p.status, false);
            }
        }
    } else if (warp == kDecMmaWarp) {
        // the whole warp runs the issuing loop; one elected lane issues each MMA and commit
        if (T > 0) {
            constexpr uint32_t idS =
                EB == 1 ? idesc_e4m3(DBN, DNR, false, false) : idesc_f16(kBF16, DBN, DNR, false, false);
            constexpr uint32_t idPV =
                EB == 1 ? idesc_e4m3(DD, DNR, false, true) : idesc_f16(kBF16, DD, DNR, false, true);
            auto issue_s = [&](int j) {
                const int u = ring_pos_k(j), s = u % kSlots;
                if (!dwait_warp(bar_full0 + 8 * s, (u / kSlots) & 1, abort_flag, p.status)) return false;
                tc_fence_after();
                // one K step covers 32 bytes of D: 16 elements of 16 bits, 32 of 8
                for (int kk = 0; kk < DD * EB / 32; ++kk) {
                    const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                    const uint64_t a = sw128_desc(sRing + s * kTileBytes + off, 16, 1024);
                    const uint64_t bq = sw128_desc(sQ + (kk >> 2) * kQChunk + (kk & 3) * 32, 16, 1024);
                    if constexpr (EB == 1)
                        mma_ss_f8_el(tmem + dcol_s(j & 1), a, bq, idS, kk > 0 ? 1u : 0u);
                    else
                        mma_ss_el(tmem + dcol_s(j & 1), a, bq, idS, kk > 0 ? 1u : 0u);
                }
                mma_commit_el(bar_s0 + 8 * (j & 1));
                mma_commit_el(bar_empty0 + 8 * s);
                return true;
            };
            auto issue_pv = [&](int j) {
                const int u = ring_pos_v(j, T), s = u % kSlots;
                if (!dwait_warp(bar_full0 + 8 * s, (u / kSlots) & 1, abort_flag, p.status)) return false;
                if (!dwait_warp(bar_p0 + 8 * (j & 1), (j >> 1) & 1, abort_flag, p.status)) return false;
                tc_fence_after();
                // one K step covers 32 / EB keys: that many 128-byte rows of V
                for (int kk = 0; kk < DBN * EB / 32; ++kk) {
                    const uint64_t a =
                        sw128_desc(sRing + s * kTileBytes + kk * (32 / EB) * 128, kChunkBytes, 1024);
                    const uint64_t bp = sw128_desc(sP + (j & 1) * C::kPBytes + (kk >> 2) * kQChunk + (kk & 3) * 32,
                                                   16, 1024);
                    if constexpr (EB == 1)
                        mma_ss_f8_el(tmem + kColO, a, bp, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                    else
                        mma_ss_el(tmem + kColO, a, bp, idPV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_el(bar_free0 + 8 * (j & 1));
                mma_commit_el(bar_empty0 + 8 * s);
                return true;
            };
            if constexpr (kR2) {
                // rounds of two tiles: S^T of round i into buffers 2i, 2i+1 (mod 4), one
                // score commit per round, then the value products of round i-1
                int u = 0;  // ring position, in the producer's order
                auto take = [&](int* sl) {
                    *sl = u % kSlots;
                    const bool r = dwait_warp(bar_full0 + 8 * *sl, (u / kSlots) & 1, abort_flag, p.status);
                    ++u;
                    return r;
                };
                auto round_pv = [&](int ir) {
                    if (!dwait_warp(bar_p0 + 8 * (ir & 1), (ir >> 1) & 1, abort_flag, p.status)) return false;
                    const int n = min(2, T - 2 * ir);
                    for (int a = 0; a < n; ++a) {
                        const int t = 2 * ir + a;
                        int sl;
                        if (!take(&sl)) return false;
                        tc_fence_after();
                        for (int kk = 0; kk < DBN * EB / 32; ++kk) {
                            const uint64_t av =
                                sw128_desc(sRing + sl * kTileBytes + kk * (32 / EB) * 128, kChunkBytes, 1024);
                            const uint64_t bp = sw128_desc(sP + (t & 3) * C::kPBytes + (kk >> 2) * kQChunk + (kk & 3) * 32,
                                                           16, 1024);
                            mma_ss_f8_el(tmem + kColO, av, bp, idPV, (t > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit_el(bar_empty0 + 8 * sl);
                    }
                    mma_commit_el(bar_free0 + 8 * (ir & 1));
                    return true;
                };
                const int R = (T + 1) / 2;
                bool ok = dwait_warp(bar_q, 0, abort_flag, p.status);
                for (int i = 0; ok && i < R; ++i) {
                    const int n = min(2, T - 2 * i);
                    for (int a = 0; ok && a < n; ++a) {
                        const int t = 2 * i + a;
                        int sl;
                        if (!(ok = take(&sl))) break;
                        tc_fence_after();
                        for (int kk = 0; kk < DD * EB / 32; ++kk) {
                            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
                            const uint64_t ak = sw128_desc(sRing + sl * kTileBytes + off, 16, 1024);
                            const uint64_t bq = sw128_desc(sQ + (kk >> 2) * kQChunk + (kk & 3) * 32, 16, 1024);
                            mma_ss_f8_el(tmem + 16u * (uint32_t)(t & 3), ak, bq, idS, kk > 0 ? 1u : 0u);
                        }
                        mma_commit_el(bar_empty0 + 8 * sl);
                    }
                    if (!ok) break;
                    mma_commit_el(bar_s0 + 8 * (i & 1));  // both score tiles of round i
                    if (i > 0) ok = round_pv(i - 1);
                }
                if (ok) round_pv(R - 1);
            } else {
                bool ok = dwait_warp(bar_q, 0, abort_flag, p.status);
                for (int j = 0; ok && j < T; ++j) {
                    ok = issue_s(j);
                    if (ok && j > 0) ok = issue_pv(j - 1);
                }
                if (ok) issue_pv(T - 1);
            }
            mma_commit_el(bar_o);
            dwait_warp_final(bar_o, 0, p.status);
        }
        __syncwarp();
    } else {
        // softmax: thread = key within the tile (and = head dimension for O^T)
        const int kl = threadIdx.x;  // 0..127
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float c = p.scale_log2;
        int lo[RP], hi[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const int i = (rblk * DNR + r) % p.M;
            key_range(i + sq.N - p.M, sq.N, p.causal, p.window, &lo[r], &hi[r]);
            if (r >= R) hi[r] = lo[r];  // padding rows see nothing: their scores are -inf, p = 0
        }
        float m_ref[RP], l_part[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            m_ref[r] = -INFINITY;
            l_part[r] = 0.f;
        }
        bool ok = true;
        if constexpr (kR2) {
            const int R = (T + 1) / 2;
            for (int i = 0; i < R; ++i) {
                const int n = min(2, T - 2 * i);  // tiles of this round
                if (!(ok = dwait_warp(bar_s0 + 8 * (i & 1), (i >> 1) & 1, abort_flag, p.status))) break;
                tc_fence_after();
                uint32_t sr[2][16];
#pragma unroll
                for (int e = 0; e < 16; ++e) sr[1][e] = 0u;
                tmem_ld_x16(tmem + lane_base + 16u * (uint32_t)((2 * i) & 3), sr[0]);
                if (n == 2) tmem_ld_x16(tmem + lane_base + 16u * (uint32_t)((2 * i + 1) & 3), sr[1]);
                asm volatile("tcgen05.wait::ld.sync.aligned;"
                             : "+r"(sr[0][0]), "+r"(sr[0][1]), "+r"(sr[0][2]), "+r"(sr[0][3]), "+r"(sr[0][4]),
                               "+r"(sr[0][5]), "+r"(sr[0][6]), "+r"(sr[0][7]), "+r"(sr[0][8]), "+r"(sr[0][9]),
                               "+r"(sr[0][10]), "+r"(sr[0][11]), "+r"(sr[0][12]), "+r"(sr[0][13]), "+r"(sr[0][14]),
                               "+r"(sr[0][15])::"memory");
                asm volatile(""
                             : "+r"(sr[1][0]), "+r"(sr[1][1]), "+r"(sr[1][2]), "+r"(sr[1][3]), "+r"(sr[1][4]),
                               "+r"(sr[1][5]), "+r"(sr[1][6]), "+r"(sr[1][7]), "+r"(sr[1][8]), "+r"(sr[1][9]),
                               "+r"(sr[1][10]), "+r"(sr[1][11]), "+r"(sr[1][12]), "+r"(sr[1][13]), "+r"(sr[1][14]),
                               "+r"(sr[1][15])::"memory");
                float t[2][RP];
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const int key = k0 + (2 * i + a) * DBN + kl;
#pragma unroll
                    for (int r = 0; r < RP; ++r)
                        t[a][r] = (a < n && key >= lo[r] && key < hi[r]) ? __uint_as_float(sr[a][r]) * c : -INFINITY;
                }
                // round row maxima across the 256 keys
                float* redj = red + (i & 1) * 4 * DNR;
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    float x = fmaxf(t[0][r], t[1][r]);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
                    if (lane == 0) redj[warp * DNR + r] = x;
                }
                if (lane == 0) mbar_arrive(bar_red0 + 8 * (i & 1));  // lane 0 wrote the warp's maxima
                if (!(ok = dwait_warp(bar_red0 + 8 * (i & 1), (i >> 1) & 1, abort_flag, p.status))) break;
                bool need_any = false;
                float alpha[RP];
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    alpha[r] = 1.f;
                    const float mt = fmaxf(fmaxf(redj[r], redj[DNR + r]), fmaxf(redj[2 * DNR + r], redj[3 * DNR + r]));
                    const float m_new = fmaxf(m_ref[r], mt);
                    if (m_new > m_ref[r] + kDecRescale) {
                        alpha[r] = ex2(m_ref[r] - m_new);
                        l_part[r] *= alpha[r];
                        m_ref[r] = m_new;
                        need_any = true;
                    }
                }
                // this round's P^T buffers were last read by the value products of round i-2
                if (i >= 2 && !(ok = dwait_warp(bar_free0 + 8 * (i & 1), ((i - 2) >> 1) & 1, abort_flag, p.status)))
                    break;
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    if (a >= n) break;
                    uint8_t* pbuf = smem + C::kOffP + ((2 * i + a) & 3) * C::kPBytes;
#pragma unroll
                    for (int r = 0; r < RP; ++r) {
                        const float m_use = (m_ref[r] == -INFINITY) ? 0.f : m_ref[r];
                        const float pr = ex2(t[a][r] - m_use);
                        l_part[r] += pr;
                        // P^T row r, key kl, in the 128-byte swizzle: 16-byte granule g of row r sits at g ^ (r & 7)
                        const int off = r * 128 + ((((kl >> 4) ^ (r & 7))) << 4) + (kl & 15);
                        pbuf[off] = (uint8_t)(pack_e4m3x4(pr, 0.f, 0.f, 0.f) & 0xFFu);
                    }
                }
                // lazy rescale of O^T (needs the value products of round i-1 complete)
                if (need_any && i > 0) {
                    if (!(ok = dwait_warp(bar_free0 + 8 * ((i - 1) & 1), ((i - 1) >> 1) & 1, abort_flag, p.status)))
                        break;
                    tc_fence_after();
                    uint32_t o[16];
                    tmem_ld_x16(tmem + lane_base + kColO, o);
                    asm volatile("tcgen05.wait::ld.sync.aligned;"
                                 : "+r"(o[0]), "+r"(o[1]), "+r"(o[2]), "+r"(o[3]), "+r"(o[4]), "+r"(o[5]), "+r"(o[6]),
                                   "+r"(o[7]), "+r"(o[8]), "+r"(o[9]), "+r"(o[10]), "+r"(o[11]), "+r"(o[12]),
                                   "+r"(o[13]), "+r"(o[14]), "+r"(o[15])::"memory");
#pragma unroll
                    for (int r = 0; r < RP; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
                    tmem_st_x16(tmem + lane_base + kColO, o);
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();  // every lane's P^T bytes and TMEM stores before lane 0's arrival
                if (lane == 0) mbar_arrive(bar_p0 + 8 * (i & 1));
            }
        } else {
            for (int j = 0; j < T; ++j) {
                const int key = k0 + j * DBN + kl;
                if (!(ok = dwait_warp(bar_s0 + 8 * (j & 1), (j >> 1) & 1, abort_flag, p.status))) break;
                tc_fence_after();
                uint32_t sr[16];
                tmem_ld_x16(tmem + lane_base + dcol_s(j & 1), sr);
                asm volatile("tcgen05.wait::ld.sync.aligned;"
                             : "+r"(sr[0]), "+r"(sr[1]), "+r"(sr[2]), "+r"(sr[3]), "+r"(sr[4]), "+r"(sr[5]), "+r"(sr[6]),
                               "+r"(sr[7]), "+r"(sr[8]), "+r"(sr[9]), "+r"(sr[10]), "+r"(sr[11]), "+r"(sr[12]),
                               "+r"(sr[13]), "+r"(sr[14]), "+r"(sr[15])::"memory");
                float t[RP];
#pragma unroll
                for (int r = 0; r < RP; ++r)
                    t[r] = (key >= lo[r] && key < hi[r]) ? __uint_as_float(sr[r]) * c : -INFINITY;
                // tile row maxima across the 128 keys
                float* redj = red + (j & 1) * 4 * DNR;
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    float x = t[r];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
                    if (lane == 0) redj[warp * DNR + r] = x;
                }
                if (lane == 0) mbar_arrive(bar_red0 + 8 * (j & 1));  // lane 0 wrote the warp's maxima
                if (!(ok = dwait_warp(bar_red0 + 8 * (j & 1), (j >> 1) & 1, abort_flag, p.status))) break;
                bool need_any = false;
                float alpha[RP];
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    alpha[r] = 1.f;
                    const float mt = fmaxf(fmaxf(redj[r], redj[DNR + r]), fmaxf(redj[2 * DNR + r], redj[3 * DNR + r]));
                    const float m_new = fmaxf(m_ref[r], mt);
                    if (m_new > m_ref[r] + kDecRescale) {
                        alpha[r] = ex2(m_ref[r] - m_new);
                        l_part[r] *= alpha[r];
                        m_ref[r] = m_new;
                        need_any = true;
                    }
                }
                // P^T buffer j&1 was last read by the value product of tile j-2
                if (j >= 2 && !(ok = dwait_warp(bar_free0 + 8 * (j & 1), ((j - 2) >> 1) & 1, abort_flag, p.status)))
                    break;
                uint8_t* pbuf = smem + C::kOffP + (j & 1) * C::kPBytes;
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    const float m_use = (m_ref[r] == -INFINITY) ? 0.f : m_ref[r];
                    const float pr = ex2(t[r] - m_use);
                    l_part[r] += pr;
                    // P^T row r, key kl, in the 128-byte swizzle: 16-byte granule g of row r sits at g ^ (r & 7)
                    if constexpr (EB == 1) {
                        const int off = r * 128 + ((((kl >> 4) ^ (r & 7))) << 4) + (kl & 15);
                        pbuf[off] = (uint8_t)(pack_e4m3x4(pr, 0.f, 0.f, 0.f) & 0xFFu);
                    } else {
                        const int kc = kl >> 6, k64 = kl & 63;
                        const uint32_t pk = kBF16 ? pack_bf16(pr, 0.f) : pack_f16(pr, 0.f);
                        const int off = kc * kQChunk + r * 128 + ((((k64 >> 3) ^ (r & 7))) << 4) + (k64 & 7) * 2;
                        *reinterpret_cast<uint16_t*>(pbuf + off) = (uint16_t)(pk & 0xFFFFu);
                    }
                }
                // lazy rescale of O^T (needs the value product of tile j-1 complete)
                if (need_any && j > 0) {
                    if (!(ok = dwait_warp(bar_free0 + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, p.status)))
                        break;
                    tc_fence_after();
                    uint32_t o[16];
                    tmem_ld_x16(tmem + lane_base + kColO, o);
                    asm volatile("tcgen05.wait::ld.sync.aligned;"
                                 : "+r"(o[0]), "+r"(o[1]), "+r"(o[2]), "+r"(o[3]), "+r"(o[4]), "+r"(o[5]), "+r"(o[6]),
                                   "+r"(o[7]), "+r"(o[8]), "+r"(o[9]), "+r"(o[10]), "+r"(o[11]), "+r"(o[12]),
                                   "+r"(o[13]), "+r"(o[14]), "+r"(o[15])::"memory");
#pragma unroll
                    for (int r = 0; r < RP; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
                    tmem_st_x16(tmem + lane_base + kColO, o);
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();  // every lane's P^T bytes and TMEM stores before lane 0's arrival
                if (lane == 0) mbar_arrive(bar_p0 + 8 * (j & 1));
            }

        }

        // summary of this split: m (base 2), l, acc for the group's rows
        int stop = 0;
        if (lane == 0) stop = *abort_flag ? 1 : 0;
        stop = __shfl_sync(0xffffffffu, stop, 0);
        bool have = ok && !stop && T > 0 && dwait_warp(bar_o, 0, abort_flag, p.status);
        if (have) {
            tc_fence_after();
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                if (r < R) {
                    float x = l_part[r];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                    if (lane == 0) lred[warp * DNR + r] = x;
                }
            }
            if (lane == 0) mbar_arrive(bar_lred);  // lane 0 wrote the warp's row sums
            have = dwait_warp(bar_lred, 0, abort_flag, p.status);
        }
        if (have) {
            uint32_t o[16];
            tmem_ld_x16(tmem + lane_base + kColO, o);
            asm volatile("tcgen05.wait::ld.sync.aligned;"
                         : "+r"(o[0]), "+r"(o[1]), "+r"(o[2]), "+r"(o[3]), "+r"(o[4]), "+r"(o[5]), "+r"(o[6]),
                           "+r"(o[7]), "+r"(o[8]), "+r"(o[9]), "+r"(o[10]), "+r"(o[11]), "+r"(o[12]), "+r"(o[13]),
                           "+r"(o[14]), "+r"(o[15])::"memory");
#pragma unroll
            for (int r = 0; r < RP; ++r) {
                if (r < R) {
                    const float lsum = lred[r] + lred[DNR + r] + lred[2 * DNR + r] + lred[3 * DNR + r];
                    if (p.cluster) {  // the summary stays in this CTA's (now idle) ring
                        part[r * DD + kl] = __uint_as_float(o[r]);
                        if (kl == 0) {
                            part[DNR * DD + r] = m_ref[r];
                            part[DNR * DD + DNR + r] = lsum;
                        }
                        continue;
                    }
                    const size_t slot = (size_t)(row_base + r) * p.S + split;
                    if (kl < Dh) p.ws_acc[slot * Dh + kl] = __uint_as_float(o[r]);
                    if (kl == 0) {
                        p.ws_m[slot] = m_ref[r];
                        p.ws_l[slot] = lsum;
                    }
                }
            }
        } else if (p.cluster) {
            // no key in this split (or it gave up): the empty summary
            for (int r = 0; r < R; ++r) {
                part[r * DD + kl] = 0.f;
                if (kl == 0) {
                    part[DNR * DD + r] = -INFINITY;
                    part[DNR * DD + DNR + r] = 0.f;
                }
            }
        } else {
            // no key of this split, or it gave up on a bounded wait: the empty
            // summary, so the merge never reads a slot this call did not write
            for (int r = 0; r < R; ++r) {
                const size_t slot = (size_t)(row_base + r) * p.S + split;
                if (kl < Dh) p.ws_acc[slot * Dh + kl] = 0.f;
                if (kl == 0) {
                    p.ws_m[slot] = -INFINITY;
                    p.ws_l[slot] = 0.f;
                }
            }
        }
    }

    if (p.cluster) {
        // every thread of every CTA of the cluster reaches this point (all waits
        // above are bounded), so the cluster barriers complete
        cluster_sync_all();
        if (warp < 4) {
            // rank s merges rows s, s + S, ...; thread kl = head dimension d: the
            // common-maximum merge of the S summaries (maxima in base 2), one cast.
            // All S summaries of a row are loaded before any is used, so the
            // distributed-shared-memory round trips overlap.
            const int kl = threadIdx.x;
            const uint32_t local = smem_u32(part);
            for (int r = (int)cluster_rank(); r < R; r += p.S) {
                float ms[kMaxClusterSplits], ls[kMaxClusterSplits], as[kMaxClusterSplits];
#pragma unroll
                for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
                    ms[sp] = -INFINITY;
                    ls[sp] = 0.f;
                    as[sp] = 0.f;
                    if (sp < p.S) {
                        const uint32_t base = map_to_rank(local, sp);
                        ms[sp] = ld_cluster_f32(base + 4u * (DNR * DD + r));
                        ls[sp] = ld_cluster_f32(base + 4u * (DNR * DD + DNR + r));
                        as[sp] = ld_cluster_f32(base + 4u * (r * DD + kl));
                    }
                }
                float mx = -INFINITY;
#pragma unroll
                for (int sp = 0; sp < kMaxClusterSplits; ++sp) mx = fmaxf(mx, ms[sp]);
                float L = 0.f, x = 0.f;
#pragma unroll
                for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
                    const float w = (ms[sp] == -INFINITY) ? 0.f : exp2f(ms[sp] - mx);  // an empty summary weighs 0
                    L = fmaf(w, ls[sp], L);
                    x = fmaf(w, as[sp], x);
                }
                x *= L > 0.f ? p.out_scale / L : 0.f;
                const size_t out = (size_t)(row_base + r) * Dh + kl;
                if (kl >= Dh) {
                } else if (p.out_dtype == ATTN_BF16) {
                    reinterpret_cast<uint16_t*>(p.o)[out] = (uint16_t)(pack_bf16(x, 0.f) & 0xFFFFu);
                } else {
                    reinterpret_cast<uint16_t*>(p.o)[out] = (uint16_t)(pack_f16(x, 0.f) & 0xFFFFu);
                }
                if (kl == 0 && p.lse) p.lse[row_base + r] = L > 0.f ? (mx + log2f(L)) * kLn2 : -INFINITY;
            }
        }
        // every CTA keeps its shared memory until the others have read it
        cluster_sync_relaxed();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kDecMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kCols);
    }
}

int sm_count() {
    const int n = device_sm_count();
    return n > 0 ? n : 148;
}

template <int EB, bool kBF16, int RP, bool kPaged>
cudaError_t launch_decode_t(const Problem& pr, const void* q, const void* k, const void* v, const PagedKV* kv,
                            int chunk, int S, const SplitWorkspace& ws, int* status, cudaStream_t stream,
                            DecodeOut* out) {
    static PerDeviceOnce attr_once;
    const cudaError_t attr_err = once_per_device(attr_once, [] {
        return cudaFuncSetAttribute(attn_decode_kernel<EB, kBF16, RP, kPaged>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<EB>::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tq, tk, tv;
    // D = 64 (16-bit): the maps' rows are 64 elements, so the second 64-column box of
    // every Q, K and V tile lies past the row and reads as zeros; the products then
    // run as for D = 128 (the zero half adds nothing to the scores, and the upper
    // 64 rows of O^T stay zero and are never written out).
    if (EB == 1 && pr.D != DD) return cudaErrorInvalidValue;
    if (!make_tensor_map(&tq, q, pr.D, pr.B * pr.Hq * pr.M, 1, DNR, kBF16, EB)) return cudaErrorInvalidValue;
    if (kPaged) {
        const int box = kv->page_size < DBN ? kv->page_size : DBN;
        if (!make_tensor_map(&tk, kv->k_pages, pr.D, kv->page_size, kv->num_pages * pr.Hkv, box, kBF16, EB) ||
            !make_tensor_map(&tv, kv->v_pages, pr.D, kv->page_size, kv->num_pages * pr.Hkv, box, kBF16, EB))
            return cudaErrorInvalidValue;
    } else if (!make_tensor_map(&tk, k, pr.D, pr.N, pr.B * pr.Hkv, DBN, kBF16, EB) ||
               !make_tensor_map(&tv, v, pr.D, pr.N, pr.B * pr.Hkv, DBN, kBF16, EB)) {
        return cudaErrorInvalidValue;
    }
    DecodeParams dp = {};
    dp.ws_m = ws.m;
    dp.ws_l = ws.l;
    dp.ws_acc = ws.acc;
    dp.status = status;
    dp.Hq = pr.Hq;
    dp.Hkv = pr.Hkv;
    dp.M = pr.M;
    dp.N = pr.N;
    dp.G = pr.G;
    dp.R = pr.G * pr.M;
    dp.D = pr.D;
    dp.causal = pr.causal;
    dp.window = pr.window;
    dp.scale_log2 = pr.scale_log2;
    dp.klo = pr.klo;
    dp.khi = pr.khi;
    dp.kbase = split_base(pr);
    dp.chunk = chunk;
    dp.S = S;
    if (kPaged) {
        dp.block_table = kv->block_table;
        dp.seq_lens = kv->seq_lens;
        dp.page_size = kv->page_size;
        dp.max_pages = kv->max_pages;
        dp.max_len = kv->max_len;
        dp.oob_z = kv->num_pages * pr.Hkv;
    }
    // Up to 8 splits of a group form one cluster and merge in the kernel
    const bool cluster = out && out->o && S <= kMaxClusterSplits;
    if (cluster) {
        dp.cluster = 1;
        dp.o = out->o;
        dp.lse = out->lse;
        dp.out_dtype = pr.dtype;
        dp.out_scale = out->out_scale;
    }
    // Programmatic launch: CTAs may start their setup (barriers, TMEM) while the
    // previous kernel in the stream drains; griddepcontrol.wait orders the rest.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S, pr.B * pr.Hkv, (pr.G * pr.M + DNR - 1) / DNR);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = DCfg<EB>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_decode_kernel<EB, kBF16, RP, kPaged>, tq, tk, tv, dp);
    if (out) out->merged = cluster && e == cudaSuccess;
    return e;
}

// e4m3: 8-bit inputs (the problem's dtype is then the output type, which the
// split kernel never writes)
template <bool kPaged>
cudaError_t launch_decode_any(const Problem& p, const void* q, const void* k, const void* v, const PagedKV* kv,
                              int chunk, int S, const SplitWorkspace& ws, int* status, cudaStream_t stream,
                              DecodeOut* out, bool e4m3 = false) {
    const int R = p.G * p.M;
    if (e4m3) {
        if (R <= 4) return launch_decode_t<1, true, 4, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out);
        if (R <= 8) return launch_decode_t<1, true, 8, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out);
        return launch_decode_t<1, true, 16, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out);
    }
    const bool bf = p.dtype == ATTN_BF16;
    if (R <= 4) return bf ? launch_decode_t<2, true, 4, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out)
                          : launch_decode_t<2, false, 4, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out);
    if (R <= 8) return bf ? launch_decode_t<2, true, 8, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out)
                          : launch_decode_t<2, false, 8, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out);
    return bf ? launch_decode_t<2, true, 16, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out)
              : launch_decode_t<2, false, 16, kPaged>(p, q, k, v, kv, chunk, S, ws, status, stream, out);
}

// Splits of `tiles` key tiles over `groups` KV groups: every CTA resident at
// once when possible (per_sm per SM), each streaming an equal run of tiles.
void plan_splits(int tiles, int groups, int* chunk, int* S, int per_sm) {
    const int slots = per_sm * sm_count();
    int s = groups > 0 ? slots / groups : 1;
    if (s < 1) s = 1;
    if (s > tiles) s = tiles;
    if (s > 4096) s = 4096;
    const int per = (tiles + s - 1) / s;
    *chunk = per * DBN;
    *S = (tiles + per - 1) / per;
}

}  // namespace

// D = 128, or 64 with 16-bit inputs (the 8-bit entry points take D = 128 only);
// any number of grouped rows: CTAs of 16 rows each along the grid's z (at most 65535).
bool decode_tc_supported(const Problem& p) {
    return (p.D == DD || p.D == 64) && p.B * p.Hkv <= 65535 && ((long long)p.G * p.M + DNR - 1) / DNR <= 65535;
}

// (KV group, block of 16 grouped rows) pairs: the CTAs of one split
static int row_groups(const Problem& p) { return p.B * p.Hkv * ((p.G * p.M + DNR - 1) / DNR); }

// CTAs resident per SM (two for both input widths; the plan keeps the 8-bit
// switch so that its workspace query stays separate from the 16-bit one)
int ctas_per_sm(const Problem& p, bool e4m3) {
    (void)p;
    (void)e4m3;
    return 2;
}

int decode_plan_tc(const Problem& p, int* chunk, int* S, bool e4m3) {
    const int kbase = split_base(p);
    const int tiles = p.khi > kbase ? (p.khi - kbase + DBN - 1) / DBN : 1;
    plan_splits(tiles, row_groups(p), chunk, S, ctas_per_sm(p, e4m3));
    return ATTN_OK;
}

cudaError_t launch_decode_tc(const Problem& p, const void* q, const void* k, const void* v, int chunk, int S,
                             const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out) {
    return launch_decode_any<false>(p, q, k, v, nullptr, chunk, S, ws, status, stream, out);
}

// Paged: the plan must cover any sequence up to kv.max_len keys. Without a
// window a sequence's range starts at key 0; with one it spans at most
// window + M - 1 keys from an unaligned start.
int decode_plan_paged(const Problem& p, const PagedKV& kv, int* chunk, int* S, bool e4m3) {
    const int len_tiles = (kv.max_len + DBN - 1) / DBN;
    int tiles = len_tiles;
    if (p.window > 0) {
        const long long span = (long long)p.window + p.M - 1 + (DBN - 1);
        const long long wt = (span + DBN - 1) / DBN;
        if (wt < tiles) tiles = (int)wt;
    }
    if (tiles < 1) tiles = 1;
    plan_splits(tiles, row_groups(p), chunk, S, ctas_per_sm(p, e4m3));
    return ATTN_OK;
}

cudaError_t launch_decode_paged(const Problem& p, const void* q, const PagedKV& kv, int chunk, int S,
                                const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out,
                                bool e4m3) {
    return launch_decode_any<true>(p, q, nullptr, nullptr, &kv, chunk, S, ws, status, stream, out, e4m3);
}

cudaError_t launch_decode_e4m3(const Problem& p, const void* q, const void* k, const void* v, int chunk, int S,
                               const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out) {
    return launch_decode_any<false>(p, q, k, v, nullptr, chunk, S, ws, status, stream, out, true);
}

}  // namespace attn
