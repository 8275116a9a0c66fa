// Split-KV decode that allocates nothing.
//
// Some callers cannot allocate device memory at the moment they need the
// forward: an allocator hook or custom memory pool that must not re-enter
// cudaMalloc, a real-time or driver-level caller that forbids allocation on
// its hot path, or code that runs where the CUDA caching allocator is not
// available. For them, attn_fwd_decode_noalloc runs the same split-KV kernel
// and merge kernel as the decode path of attn_fwd_ex, but keeps the partial
// (m, l, acc) summaries in one fixed device array declared below instead of a
// caller- or library-allocated workspace.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it. Host code may not pass the symbol itself to a kernel: on the host
// it names a stand-in, not a device address. Its device address is looked up
// once per device with cudaGetSymbolAddress (while that device is current)
// and cached.
#include <mutex>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call for that device); nullptr on failure.
void* scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                                       int Hkv, int M, int N, int D, int causal, int window, float scale,
                                       attn_dtype_t dtype, void* stream) {
    Problem p;
    int rc = validate_problem(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    if (!decode_supported(p)) return ATTN_ERR_HEADDIM;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((int64_t)p.B * p.Hq * p.M == 0) return ATTN_OK;
    if (p.N == 0) {  // every row sees no key: output 0
        const size_t bytes = (size_t)p.B * p.Hq * p.M * p.D * 2;
        return cudaMemsetAsync(o, 0, bytes, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    if (!decode_tc_supported(p) && !simt_grid_ok(p)) return ATTN_ERR_PATH;
    int chunk = 0, S = 0;
    rc = decode_plan(p, &chunk, &S);
    if (rc != ATTN_OK) return rc;
    const int rows = p.B * p.Hq * p.M;
    // With at most kMaxClusterSplits splits per KV head the tcgen05 split kernel
    // merges them inside its thread-block cluster and never touches the array,
    // so only the other plans are limited by the array's size.
    const bool in_cluster = decode_tc_supported(p) && S <= kMaxClusterSplits;
    if (!in_cluster && split_workspace_bytes(rows, S, p.D) > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
    int* status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    // Every (row, split) summary the merge reads is written by the split
    // kernel of this same call (an empty one where a split sees no key or
    // gives up), so nothing has to be cleared first.
    SplitWorkspace w{nullptr, nullptr, nullptr};
    if (!in_cluster) {
        void* base = scratch_ptr();
        if (!base) return ATTN_ERR_CUDA;
        w = split_workspace(base, rows, S, p.D);
    }
    DecodeOut out{o, nullptr, 1.0f, false};
    if (launch_decode(p, q, k, v, chunk, S, w, status, s, &out) != cudaSuccess) return ATTN_ERR_CUDA;
    if (out.merged) return ATTN_OK;
    if (launch_merge(w.m, w.l, w.acc, o, nullptr, nullptr, nullptr, rows, S, p.D, p.dtype, 1.0f, true, s) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    return ATTN_OK;
}
