// Internal declarations shared by the CUDA sources of the library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "attn.h"

namespace attn {

// ---- per-device host state -------------------------------------------------
// Kernel attributes (the dynamic shared-memory limit) and cached device
// properties belong to one device; each is set up once per device, on the
// first launch with that device current, so one process may drive several GPUs.
constexpr int kMaxDevices = 64;

struct PerDeviceOnce {
    std::atomic<uint64_t> done{0};  // bit d: set up on device d
    std::mutex mu;
};

// Runs fn() (returning cudaError_t) once per device: on the first call with that
// device current. A failure is returned and not cached, so a later call retries.
template <class F>
cudaError_t once_per_device(PerDeviceOnce& o, F&& fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (o.done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    std::lock_guard<std::mutex> lock(o.mu);
    if (o.done.load(std::memory_order_relaxed) & bit) return cudaSuccess;
    const cudaError_t e = fn();
    if (e == cudaSuccess) o.done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Number of SMs of the current device (cached per device); 0 when it cannot be read.
int device_sm_count();

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// One forward problem, validated. Positions follow the bottom-right rule
// p_i = i + N - M; klo/khi bound the keys that any row of the problem may see.
struct Problem {
    int B, Hq, Hkv, M, N, D;
    int causal, window;
    float scale;       // logit scale (resolved: never 0)
    float scale_log2;  // scale * log2(e): logits are handled in base 2
    int dtype;         // ATTN_BF16 / ATTN_FP16
    int G;             // Hq / Hkv
    int klo, khi;      // union of the visible key ranges over all rows
    float* lse;        // optional [B*Hq*M] natural-log sum of exp of the logits (nullptr: not written)
};

// Keys [lo, hi) visible to the query at position p (hi <= lo: none).
__host__ __device__ inline void key_range(int p, int N, int causal, int window, int* lo, int* hi) {
    int h = causal ? (p + 1 < N ? p + 1 : N) : N;
    int l = (window > 0) ? (p - window + 1 > 0 ? p - window + 1 : 0) : 0;
    if (h < 0) h = 0;
    *lo = l;
    *hi = h;
}

// The CUDA-core kernel (the SIMT path, and split decode of shapes the tcgen05
// split kernel does not take) runs one (batch, query head) per grid y index,
// whose limit is 65535.
inline bool simt_grid_ok(const Problem& p) { return (long long)p.B * p.Hq <= 65535; }

// Split-KV workspace: the union key range [klo, khi) is cut into S chunks of
// `chunk` keys (a multiple of 128) starting at split_base(p); partial summaries are [rows][S] floats m and l (m in base-2
// logit units) and [rows][S][D] floats acc. Each part is 256-byte aligned.
// Splits start at the visible range's start rounded down to a 128-key tile.
inline int split_base(const Problem& p) { return (p.klo / 128) * 128; }

struct SplitWorkspace {
    float* m;
    float* l;
    float* acc;
};
size_t split_workspace_bytes(int rows, int S, int D);
SplitWorkspace split_workspace(void* base, int rows, int S, int D);

// Launchers (all asynchronous on `stream`; return a CUDA error).
cudaError_t launch_simt(const Problem& p, const void* q, const void* k, const void* v, void* o,
                        int chunk, int S, const SplitWorkspace* ws, cudaStream_t stream);
cudaError_t launch_merge(const float* m, const float* l, const float* acc, void* o, float* m_out,
                         float* l_out, float* lse_out, int rows, int S, int D, int out_dtype, float unit,
                         bool programmatic, cudaStream_t stream, float out_scale = 1.0f);
// Where the split kernel may write the final output itself: when the splits of
// a group fit one thread-block cluster (S <= kMaxClusterSplits) the kernel merges
// them in the cluster and sets `merged`; otherwise the caller runs launch_merge.
constexpr int kMaxClusterSplits = 8;
struct DecodeOut {
    void* o;           // [rows][D] of p.dtype (nullptr: never merge in the kernel)
    float* lse;        // optional [rows] natural-log log-sum-exp
    float out_scale;   // multiplies the merged output (V dequantization factor, else 1)
    bool merged;       // set by the launch
};
cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v,
                          int chunk, int S, const SplitWorkspace& ws, int* status,
                          cudaStream_t stream, DecodeOut* out = nullptr);
bool decode_supported(const Problem& p);
int decode_plan(const Problem& p, int* chunk, int* S);
// tcgen05 split kernel (D = 128, or 64 for 16-bit inputs; grouped rows per KV head in CTAs of 16)
bool decode_tc_supported(const Problem& p);
// e4m3: the plan of the 8-bit kernel (more CTAs per SM, so more splits)
int decode_plan_tc(const Problem& p, int* chunk, int* S, bool e4m3 = false);
cudaError_t launch_decode_tc(const Problem& p, const void* q, const void* k, const void* v, int chunk, int S,
                             const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out = nullptr);

// Paged KV cache (decode): pools [num_pages][Hkv][page_size][D]; sequence b's
// key j lives in row j % page_size of page block_table[b * max_pages + j / page_size];
// sequence b holds min(seq_lens[b], max_len) keys.
struct PagedKV {
    const void* k_pages;
    const void* v_pages;
    const int* block_table;
    const int* seq_lens;
    int num_pages, page_size, max_pages, max_len;
};
int decode_plan_paged(const Problem& p, const PagedKV& kv, int* chunk, int* S, bool e4m3 = false);
// e4m3: Q and the pools hold E4M3 bytes (p.scale_log2 then includes the Q and K
// dequantization factors; the merge applies V's)
cudaError_t launch_decode_paged(const Problem& p, const void* q, const PagedKV& kv, int chunk, int S,
                                const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out = nullptr,
                                bool e4m3 = false);
// Which kernel takes a paged call: the tcgen05 split kernel (D = 128; D = 64 for
// 16-bit caches), else the grouped CUDA-core kernel (D in {16, 32, 64}; grouped
// rows up to 8 * 65535).
bool paged_tc_supported(const Problem& p, bool e4m3);
bool paged_group_supported(const Problem& p);
int paged_group_plan(const Problem& p, const PagedKV& kv, int* chunk, int* S);
// ws may be null when S == 1 (the kernel then writes o, times out_scale);
// otherwise the caller merges the summaries. e4m3: Q and the pools hold E4M3
// bytes and p.dtype is the output type.
cudaError_t launch_paged_group(const Problem& p, const void* q, const PagedKV& kv, int chunk, int S,
                               const SplitWorkspace* ws, void* o, float out_scale, bool e4m3,
                               cudaStream_t stream);
// The tcgen05 split kernel on contiguous E4M3 inputs (same plan as launch_decode_tc)
cudaError_t launch_decode_e4m3(const Problem& p, const void* q, const void* k, const void* v, int chunk, int S,
                               const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out = nullptr);

// Backward pass (tcgen05, D in {64, 128}): the caller's tensors, device pointers.
struct BwdArgs {
    const void *q, *k, *v, *o, *d_o;
    const float* lse;  // [B*Hq*M], natural log, from the forward
    void *dq, *dk, *dv;
};
size_t bwd_workspace_bytes(int B, int Hq, int M);
cudaError_t launch_bwd(const Problem& p, const BwdArgs& a, void* ws, int* status, cudaStream_t stream);

// Wide-row split softmax (three kernels, scratch [M][T + 1] float2)
bool split_softmax_chunk_ok(int chunk);
size_t split_softmax_ws_bytes(int M, int N, int chunk);
cudaError_t launch_split_softmax(const void* x, void* y, int M, int N, int chunk, int dtype, void* ws,
                                 cudaStream_t stream);

// Metadata validation and the device status word, shared by every entry point.
int validate_problem(const void* q, const void* k, const void* v, const void* o, int B, int Hq, int Hkv, int M,
                     int N, int D, int causal, int window, float scale, int dtype, Problem* p);
int* device_status_ptr();

// tcgen05 prefill: returns ATTN_OK, ATTN_ERR_PATH (cannot run this problem)
// or ATTN_ERR_CUDA.
int launch_prefill(const Problem& p, const void* q, const void* k, const void* v, void* o,
                   int* status, cudaStream_t stream);
bool prefill_supported(const Problem& p);
// The pair-MMA prefill (tcgen05 cta_group::2, clusters of two CTAs), D = 128,
// 16-bit inputs: returns ATTN_OK, ATTN_ERR_HEADDIM or ATTN_ERR_CUDA.
int launch_prefill_pair(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                        cudaStream_t stream);
bool prefill_pair_supported(const Problem& p);
// The prefill kernel with one P-ready arrival withheld (failure-path self-test;
// D = 128): its bounded waits run out and every CTA takes the abort path.
int launch_prefill_withheld(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                            long withhold_p_at, cudaStream_t stream);
// The same kernel on E4M3 inputs (D = 128, or 64 read as 128 with the upper
// half zero); p.dtype is the output type and
// p.scale_log2 already includes the Q and K dequantization factors.
int launch_prefill_e4m3(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                        float v_scale, cudaStream_t stream);

}  // namespace attn
