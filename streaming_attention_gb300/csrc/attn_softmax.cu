// Wide-row split softmax: softmax over each row of a [M, N] matrix whose rows
// are too wide for one block ("Intermediate and advanced kernel workshops",
// workshop A2: three ordered kernels with per-call scratch; answer key, A2 row:
// partial statistics per chunk, a merge rescaled to the common maximum, then a
// reread that normalizes, ordered by one stream).
//
//   1. attn_softmax_stats_kernel: one block per (row, chunk of C columns) keeps
//      the chunk in registers, takes its maximum and its sum of exponentials and
//      writes the partial summary (m, l) (maxima in base 2).
//   2. attn_softmax_merge_kernel: one warp per row combines the row's T partial
//      summaries relative to their common maximum (the A1 merge rule).
//   3. attn_softmax_norm_kernel: one block per (row, chunk) rereads its chunk and
//      writes y = 2^(x log2 e - m) / l, one cast.
// Scratch: [M][T + 1] (m, l) float pairs, the merged pair last (8 M (T + 1)
// bytes, T = ceil(N / C)). Padded columns of the last chunk take -inf in the
// maximum and 0 in the sum ("Kernel Notes & Checklist", gotchas ledger).
//
// Row-resident form (chunk 0): the same three steps with the reread served on
// chip. The T <= 8 chunks of a row (256 * VPT columns each) are the CTAs of one
// thread-block cluster; each keeps its chunk in registers, publishes its (m, l)
// in shared memory, reads its peers' pairs through distributed shared memory,
// merges them to the common maximum and normalizes its chunk from registers.
// x is read once and y written once; no scratch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kSmThreads = 256;

template <typename T>
__device__ __forceinline__ float sm_load(const void* p, size_t i);
template <>
__device__ __forceinline__ float sm_load<float>(const void* p, size_t i) {
    return __ldg(static_cast<const float*>(p) + i);
}
template <>
__device__ __forceinline__ float sm_load<__nv_bfloat16>(const void* p, size_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}
template <>
__device__ __forceinline__ float sm_load<__half>(const void* p, size_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
}
template <typename T>
__device__ __forceinline__ void sm_store(void* p, size_t i, float v);
template <>
__device__ __forceinline__ void sm_store<float>(void* p, size_t i, float v) {
    static_cast<float*>(p)[i] = v;
}
template <>
__device__ __forceinline__ void sm_store<__nv_bfloat16>(void* p, size_t i, float v) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}
template <>
__device__ __forceinline__ void sm_store<__half>(void* p, size_t i, float v) {
    static_cast<__half*>(p)[i] = __float2half_rn(v);
}

// W consecutive elements starting at element i (i a multiple of W, the address
// W * sizeof(T) aligned), as floats; and the matching store.
template <typename T, int W>
__device__ __forceinline__ void vload(const void* p, size_t i, float (&v)[W]) {
    if constexpr (sizeof(T) == 4) {
        static_assert(W == 4, "fp32 vectors are 4 wide");
        const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
        v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
    } else {
        uint32_t w[W / 2];
        if constexpr (W == 8) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + i));
            w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w;
        } else {
            static_assert(W == 4, "16-bit vectors are 4 or 8 wide");
            const uint2 a = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i));
            w[0] = a.x, w[1] = a.y;
        }
#pragma unroll
        for (int k = 0; k < W / 2; ++k) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                v[2 * k] = __uint_as_float(w[k] << 16);
                v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            } else {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
                v[2 * k] = f.x, v[2 * k + 1] = f.y;
            }
        }
    }
}
template <typename T, int W>
__device__ __forceinline__ void vstore(void* p, size_t i, const float (&v)[W]) {
    if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        uint32_t w[W / 2];
#pragma unroll
        for (int k = 0; k < W / 2; ++k) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            } else {
                const __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
                w[k] = *reinterpret_cast<const uint32_t*>(&h);
            }
        }
        if constexpr (W == 8)
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p) + i) = make_uint4(w[0], w[1], w[2], w[3]);
        else
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + i) = make_uint2(w[0], w[1]);
    }
}
template <typename T, int CPT>
struct VecW {  // vector width in elements for CPT columns per thread
    static constexpr int kMax = 16 / (int)sizeof(T);
    static constexpr int value = CPT < kMax ? CPT : kMax;
};

// Block-wide maximum / sum of one value per thread (256 threads).
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, w) : v + w;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read by a previous reduction
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[lane & 7];
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = kMax ? fmaxf(v, w) : v + w;
    }
    return v;
}

// Column of element k (of CPT) of this thread within its chunk: vectors of W
// consecutive columns, consecutive threads on consecutive vectors (coalesced).
template <int CPT, int W>
__device__ __forceinline__ int chunk_col(int k) {
    return ((k / W) * kSmThreads + (int)threadIdx.x) * W + (k % W);
}

// CPT: columns of a chunk per thread (C / 256). kVec: rows are W-aligned (N % W == 0).
template <typename T, int CPT, bool kVec>
__global__ void __launch_bounds__(kSmThreads) attn_softmax_stats_kernel(const void* x, float2* ws, int N, int T_) {
    constexpr int W = kVec ? VecW<T, CPT>::value : 1;
    __shared__ float red[8];
    const int chunk = blockIdx.x, row = blockIdx.y;
    const size_t base = (size_t)row * N;
    const int c0 = chunk * CPT * kSmThreads;
    float t[CPT];
    float mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < CPT / W; ++v) {
        const int col = c0 + chunk_col<CPT, W>(v * W);
        float e[W];
        if (col < N) {  // with kVec, N % W == 0: the whole vector is in the row
            if constexpr (W > 1)
                vload<T, W>(x, base + col, e);
            else
                e[0] = sm_load<T>(x, base + col);
        }
#pragma unroll
        for (int k = 0; k < W; ++k) {
            t[v * W + k] = col < N ? e[k] * kLog2e : -INFINITY;  // padding: -inf for the max
            mx = fmaxf(mx, t[v * W + k]);
        }
    }
    mx = block_reduce<true>(mx, red);  // finite: every chunk holds at least one column
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < CPT; ++k) s += exp2f(t[k] - mx);  // padding contributes 0 to the sum
    s = block_reduce<false>(s, red);
    if (threadIdx.x == 0) ws[(size_t)row * (T_ + 1) + chunk] = make_float2(mx, s);
}

__global__ void __launch_bounds__(kSmThreads) attn_softmax_merge_kernel(float2* ws, int M, int T_) {
    const int row = blockIdx.x * (kSmThreads / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= M) return;
    float2* r = ws + (size_t)row * (T_ + 1);
    float mx = -INFINITY;
    for (int t = lane; t < T_; t += 32) mx = fmaxf(mx, r[t].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float l = 0.f;
    for (int t = lane; t < T_; t += 32) {
        const float2 ml = r[t];
        l += ml.x == -INFINITY ? 0.f : ml.y * exp2f(ml.x - mx);  // an empty summary weighs 0
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) r[T_] = make_float2(mx, l);
}

template <typename T, int CPT, bool kVec>
__global__ void __launch_bounds__(kSmThreads)
    attn_softmax_norm_kernel(const void* x, void* y, const float2* ws, int N, int T_) {
    constexpr int W = kVec ? VecW<T, CPT>::value : 1;
    const int chunk = blockIdx.x, row = blockIdx.y;
    const size_t base = (size_t)row * N;
    const float2 ml = ws[(size_t)row * (T_ + 1) + T_];
    const float inv = 1.f / ml.y;
    const int c0 = chunk * CPT * kSmThreads;
#pragma unroll
    for (int v = 0; v < CPT / W; ++v) {
        const int col = c0 + chunk_col<CPT, W>(v * W);
        if (col >= N) continue;
        float e[W];
        if constexpr (W > 1) {
            vload<T, W>(x, base + col, e);
#pragma unroll
            for (int k = 0; k < W; ++k) e[k] = exp2f(e[k] * kLog2e - ml.x) * inv;
            vstore<T, W>(y, base + col, e);
        } else {
            sm_store<T>(y, base + col, exp2f(sm_load<T>(x, base + col) * kLog2e - ml.x) * inv);
        }
    }
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The closing barrier orders nothing in memory (the remote reads it protects have
// returned their values): a relaxed arrival does not wait for this CTA's global
// stores to complete, as a release would.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
}

// 16 raw bytes -> W floats (W = 16 / sizeof(T))
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& a, float (&v)[16 / sizeof(T)]) {
    if constexpr (sizeof(T) == 4) {
        v[0] = __uint_as_float(a.x), v[1] = __uint_as_float(a.y), v[2] = __uint_as_float(a.z),
        v[3] = __uint_as_float(a.w);
    } else {
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                v[2 * k] = __uint_as_float(w[k] << 16);
                v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            } else {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
                v[2 * k] = f.x, v[2 * k + 1] = f.y;
            }
        }
    }
}

// Chunk blockIdx.x (= cluster rank) of row blockIdx.y; gridDim.x chunks per row.
// kVec (N a multiple of 16 / sizeof(T)): each thread keeps its VPT values as the
// raw 16-byte vectors it loaded (VPT * sizeof(T) / 4 registers) and widens them
// in each pass; otherwise VPT floats.
template <typename T, int VPT, bool kVec>
__global__ void __launch_bounds__(kSmThreads, 3) attn_softmax_resident_kernel(const void* x, void* y, int N) {
    constexpr int W = kVec ? 16 / (int)sizeof(T) : 1;
    constexpr int NV = VPT / W;  // vectors (or scalars) per thread
    __shared__ float red[8];
    __shared__ float2 part;  // this chunk's (m, l), read by the whole cluster
    const int chunk = blockIdx.x, row = blockIdx.y, T_ = gridDim.x;
    const size_t base = (size_t)row * N;
    const int c0 = chunk * VPT * kSmThreads;
    using Raw = typename std::conditional<kVec, uint4, float>::type;
    Raw raw[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int col = c0 + chunk_col<VPT, W>(v * W);
        if constexpr (kVec) {
            // with kVec the whole vector is in the row or wholly past it
            raw[v] = col < N ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(x) + base + col))
                             : make_uint4(0, 0, 0, 0);
        } else {
            raw[v] = col < N ? sm_load<T>(x, base + col) : 0.f;
        }
    }
    // the values of vector v, times log2 e; padding columns -inf
    auto values = [&](int v, float (&t)[W]) {
        const int col = c0 + chunk_col<VPT, W>(v * W);
        if constexpr (kVec) {
            unpack16<T>(raw[v], t);
        } else {
            t[0] = raw[v];
        }
#pragma unroll
        for (int k = 0; k < W; ++k) t[k] = col < N ? t[k] * kLog2e : -INFINITY;
    };
    float mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float t[W];
        values(v, t);
#pragma unroll
        for (int k = 0; k < W; ++k) mx = fmaxf(mx, t[k]);
    }
    mx = block_reduce<true>(mx, red);  // finite: every chunk holds at least one column
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float t[W];
        values(v, t);
#pragma unroll
        for (int k = 0; k < W; ++k) s += exp2f(t[k] - mx);
    }
    s = block_reduce<false>(s, red);
    if (threadIdx.x == 0) part = make_float2(mx, s);
    cluster_sync_all();
    // merge of the row's T pairs relative to their common maximum (the A1 rule)
    const uint32_t local = (uint32_t)__cvta_generic_to_shared(&part);
    float2 pr[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        pr[r] = make_float2(-INFINITY, 0.f);
        if (r < T_) {
            uint32_t a;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(r));
            asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(pr[r].x), "=f"(pr[r].y) : "r"(a) : "memory");
        }
    }
    float gm = -INFINITY;
#pragma unroll
    for (int r = 0; r < 8; ++r) gm = fmaxf(gm, pr[r].x);
    float L = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) L += pr[r].x == -INFINITY ? 0.f : pr[r].y * exp2f(pr[r].x - gm);
    const float inv = 1.f / L;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int col = c0 + chunk_col<VPT, W>(v * W);
        if (col >= N) continue;
        float t[W];
        values(v, t);
#pragma unroll
        for (int k = 0; k < W; ++k) t[k] = exp2f(t[k] - gm) * inv;
        if constexpr (kVec)
            vstore<T, W>(y, base + col, t);
        else
            sm_store<T>(y, base + col, t[0]);
    }
    cluster_sync_relaxed();  // every CTA keeps its pair until the whole cluster has read it
}

// Rows of at most 8 chunks: VPT = 16 up to 32768 columns, 64 up to 131072.
template <typename T, int VPT>
cudaError_t launch_resident_t(const void* x, void* y, int M, int N, cudaStream_t stream) {
    const int C = VPT * kSmThreads, T_ = (N + C - 1) / C;
    const bool vec = N % (16 / (int)sizeof(T)) == 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T_, M);
    cfg.blockDim = dim3(kSmThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)T_;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec) return cudaLaunchKernelEx(&cfg, attn_softmax_resident_kernel<T, VPT, true>, x, y, N);
    return cudaLaunchKernelEx(&cfg, attn_softmax_resident_kernel<T, VPT, false>, x, y, N);
}

template <typename T>
cudaError_t launch_resident(const void* x, void* y, int M, int N, cudaStream_t stream) {
    if (N <= 8 * 16 * kSmThreads) return launch_resident_t<T, 16>(x, y, M, N, stream);
    return launch_resident_t<T, 64>(x, y, M, N, stream);
}

template <typename T, int CPT>
cudaError_t launch_sm_t(const void* x, void* y, int M, int N, float2* ws, cudaStream_t stream) {
    const int C = CPT * kSmThreads, T_ = (N + C - 1) / C;
    const dim3 grid(T_, M);
    // vector accesses when every row starts on a vector boundary
    const bool vec = N % VecW<T, CPT>::value == 0;
    if (vec)
        attn_softmax_stats_kernel<T, CPT, true><<<grid, kSmThreads, 0, stream>>>(x, ws, N, T_);
    else
        attn_softmax_stats_kernel<T, CPT, false><<<grid, kSmThreads, 0, stream>>>(x, ws, N, T_);
    attn_softmax_merge_kernel<<<(M + 7) / 8, kSmThreads, 0, stream>>>(ws, M, T_);
    if (vec)
        attn_softmax_norm_kernel<T, CPT, true><<<grid, kSmThreads, 0, stream>>>(x, y, ws, N, T_);
    else
        attn_softmax_norm_kernel<T, CPT, false><<<grid, kSmThreads, 0, stream>>>(x, y, ws, N, T_);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_sm_c(const void* x, void* y, int M, int N, int chunk, float2* ws, cudaStream_t stream) {
    switch (chunk) {
        case 256: return launch_sm_t<T, 1>(x, y, M, N, ws, stream);
        case 1024: return launch_sm_t<T, 4>(x, y, M, N, ws, stream);
        case 4096: return launch_sm_t<T, 16>(x, y, M, N, ws, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool split_softmax_chunk_ok(int chunk) { return chunk == 0 || chunk == 256 || chunk == 1024 || chunk == 4096; }

size_t split_softmax_ws_bytes(int M, int N, int chunk) {
    if (chunk == 0) return 0;  // row-resident: no scratch
    const size_t T_ = ((size_t)N + chunk - 1) / chunk;
    return 8 * (size_t)M * (T_ + 1);
}

cudaError_t launch_split_softmax(const void* x, void* y, int M, int N, int chunk, int dtype, void* ws,
                                 cudaStream_t stream) {
    if (chunk == 0) {
        if (dtype == ATTN_FP32) return launch_resident<float>(x, y, M, N, stream);
        if (dtype == ATTN_BF16) return launch_resident<__nv_bfloat16>(x, y, M, N, stream);
        return launch_resident<__half>(x, y, M, N, stream);
    }
    float2* w = static_cast<float2*>(ws);
    if (dtype == ATTN_FP32) return launch_sm_c<float>(x, y, M, N, chunk, w, stream);
    if (dtype == ATTN_BF16) return launch_sm_c<__nv_bfloat16>(x, y, M, N, chunk, w, stream);
    return launch_sm_c<__half>(x, y, M, N, chunk, w, stream);
}

}  // namespace attn
