// C ABI entry points: metadata validation, path choice, workspace handling.
// Every step of the computation runs in the kernels of this library.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace attn {
namespace {

// Device status word, one per device: kernels set it when a bounded wait gives
// up. Every stream on the device shares it (attn_last_device_status reads and
// clears it).
__device__ int g_status_word;

PerDeviceOnce g_status_once;
int* g_status_ptr[kMaxDevices] = {};

int* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const cudaError_t e = once_per_device(g_status_once, [dev] {
        void* p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_status_word);
        if (r == cudaSuccess) g_status_ptr[dev] = static_cast<int*>(p);
        return r;
    });
    return e == cudaSuccess ? g_status_ptr[dev] : nullptr;
}

PerDeviceOnce g_sm_once;
int g_sm_count[kMaxDevices] = {};

constexpr int64_t kI32Max = 2147483647LL;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool simt_head_dim(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }

// Validates metadata only (never values) and fills the problem description.
int validate(const void* q, const void* k, const void* v, const void* o, int B, int Hq, int Hkv, int M, int N,
             int D, int causal, int window, float scale, int dtype, Problem* p) {
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
    if (B < 0 || Hq < 0 || Hkv < 0 || M < 0 || N < 0 || D <= 0) return ATTN_ERR_SHAPE;
    if (Hq > 0 && Hkv == 0) return ATTN_ERR_SHAPE;
    if (Hq > 0 && Hq % Hkv != 0) return ATTN_ERR_GQA;
    if (!simt_head_dim(D)) return ATTN_ERR_HEADDIM;
    const int64_t nq = (int64_t)B * Hq * M * D;
    const int64_t nk = (int64_t)B * Hkv * N * D;
    if (nq > kI32Max || nk > kI32Max) return ATTN_ERR_OVERFLOW;
    if ((nq > 0 && (!q || !o)) || (nk > 0 && (!k || !v))) return ATTN_ERR_NULL;
    if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) || (o && !aligned16(o)))
        return ATTN_ERR_ALIGN;
    p->B = B;
    p->Hq = Hq;
    p->Hkv = Hkv;
    p->M = M;
    p->N = N;
    p->D = D;
    p->causal = causal ? 1 : 0;
    p->window = window > 0 ? window : 0;
    p->scale = (scale == 0.0f) ? (float)(1.0 / sqrt((double)D)) : scale;
    p->scale_log2 = p->scale * kLog2e;
    p->dtype = dtype;
    p->G = Hkv > 0 ? Hq / Hkv : 1;
    // union of the visible key ranges: row 0 gives the lowest start, row M-1
    // the highest end (both bounds grow with the position)
    int lo0 = 0, hi0 = 0, lo1 = 0, hi1 = 0;
    key_range(0 + N - M, N, p->causal, p->window, &lo0, &hi0);
    key_range(M - 1 + N - M, N, p->causal, p->window, &lo1, &hi1);
    p->klo = lo0;
    p->khi = hi1 > lo0 ? hi1 : lo0;
    p->lse = nullptr;
    return ATTN_OK;
}

bool empty_output(const Problem& p) { return (int64_t)p.B * p.Hq * p.M == 0; }

int choose_path(const Problem& p, int path) {
    if (path != ATTN_PATH_AUTO) return path;
    if (decode_supported(p) && (int64_t)p.G * p.M <= 16 && (p.khi - p.klo) >= 512 &&
        (decode_tc_supported(p) || simt_grid_ok(p)))
        return ATTN_PATH_DECODE;
    if (prefill_supported(p)) return ATTN_PATH_PREFILL;
    return ATTN_PATH_SIMT;
}

size_t workspace_for(const Problem& p, int path) {
    if (path != ATTN_PATH_DECODE || !decode_supported(p)) return 0;
    int chunk = 0, S = 0;
    if (decode_plan(p, &chunk, &S) != ATTN_OK) return 0;
    return split_workspace_bytes(p.B * p.Hq * p.M, S, p.D);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

int run(const Problem& p, const void* q, const void* k, const void* v, void* o, int path, void* ws,
        size_t ws_bytes, cudaStream_t stream) {
    if (path == ATTN_PATH_PREFILL && p.D != 64 && p.D != 128) return ATTN_ERR_HEADDIM;
    if (path == ATTN_PATH_PREFILL_PAIR && p.D != 128) return ATTN_ERR_HEADDIM;
    if (path == ATTN_PATH_DECODE && !decode_supported(p)) return ATTN_ERR_HEADDIM;
    if (empty_output(p)) return ATTN_OK;
    const bool simt = p.N == 0 ? p.lse != nullptr
                               : path == ATTN_PATH_SIMT || (path == ATTN_PATH_DECODE && !decode_tc_supported(p));
    if (simt && !simt_grid_ok(p)) return ATTN_ERR_PATH;
    if (p.N == 0) {  // every row sees no key: output 0 (and a log-sum-exp of -inf)
        if (p.lse) return cuda_status(launch_simt(p, q, k, v, o, 0, 1, nullptr, stream));
        const size_t bytes = (size_t)p.B * p.Hq * p.M * p.D * 2;
        return cuda_status(cudaMemsetAsync(o, 0, bytes, stream));
    }
    int* status = status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    switch (path) {
        case ATTN_PATH_SIMT:
            return cuda_status(launch_simt(p, q, k, v, o, 0, 1, nullptr, stream));
        case ATTN_PATH_PREFILL:
            if (!prefill_supported(p)) return ATTN_ERR_PATH;
            return launch_prefill(p, q, k, v, o, status, stream);
        case ATTN_PATH_PREFILL_PAIR:
            if (!prefill_pair_supported(p)) return ATTN_ERR_PATH;
            return launch_prefill_pair(p, q, k, v, o, status, stream);
        case ATTN_PATH_DECODE: {
            int chunk = 0, S = 0;
            int rc = decode_plan(p, &chunk, &S);
            if (rc != ATTN_OK) return rc;
            const int rows = p.B * p.Hq * p.M;
            if (!ws || ws_bytes < split_workspace_bytes(rows, S, p.D)) return ATTN_ERR_WORKSPACE;
            if (!aligned16(ws)) return ATTN_ERR_ALIGN;
            SplitWorkspace w = split_workspace(ws, rows, S, p.D);
            DecodeOut out{o, p.lse, 1.0f, false};
            cudaError_t e = launch_decode(p, q, k, v, chunk, S, w, status, stream, &out);
            if (e != cudaSuccess) return ATTN_ERR_CUDA;
            if (out.merged) return ATTN_OK;
            return cuda_status(launch_merge(w.m, w.l, w.acc, o, nullptr, nullptr, p.lse, rows, S, p.D, p.dtype,
                                            1.0f, true, stream));
        }
        default:
            return ATTN_ERR_PATH;
    }
}

// ---- host-buffer entry: copies and compute pipelined over chunks ----
//
// The problem is cut into chunks of whole (batch, KV head) groups, each a
// smaller attention problem over contiguous slices of q, k, v and o. Chunk c's
// host-to-device copies run on a copy stream, its kernel on the caller's
// stream once they land, and its output copy on a second copy stream once the
// kernel is done, so copies of one chunk overlap the compute and copies of
// others. Streams and events are made once per device and reused; one host
// call at a time uses them.
constexpr int kHostChunks = 8;

struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, in[kHostChunks] = {}, done[kHostChunks] = {};
    bool ready = false;
};
std::mutex g_host_mu;
HostPipe g_host_pipe[kMaxDevices];

HostPipe* host_pipe() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    HostPipe& hp = g_host_pipe[dev];
    if (hp.ready) return &hp;
    if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) != cudaSuccess)
        return nullptr;
    for (int c = 0; c < kHostChunks; ++c)
        if (cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.done[c], cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
    hp.ready = true;
    return &hp;
}

// One chunk: batches [b0, b0 + nb) and, within them, KV heads [g0, g0 + ng)
// (either nb == 1 or all heads).
struct HostChunk {
    int b0, nb, g0, ng;
};

int host_chunks(const Problem& p, HostChunk* out) {
    int n = 0;
    if (p.B >= kHostChunks) {
        const int per = (p.B + kHostChunks - 1) / kHostChunks;
        for (int b = 0; b < p.B; b += per) out[n++] = HostChunk{b, per < p.B - b ? per : p.B - b, 0, p.Hkv};
    } else {
        int parts = kHostChunks / (p.B > 0 ? p.B : 1);
        if (parts > p.Hkv) parts = p.Hkv;
        const int per = (p.Hkv + parts - 1) / parts;
        for (int b = 0; b < p.B; ++b)
            for (int g = 0; g < p.Hkv; g += per) out[n++] = HostChunk{b, 1, g, per < p.Hkv - g ? per : p.Hkv - g};
    }
    return n;
}

int run_host_pipelined(const Problem& p, const char* q_h, const char* k_h, const char* v_h, char* o_h, char* q_d,
                       char* k_d, char* v_d, char* o_d, int path, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_host_mu);
    HostPipe* hp = host_pipe();
    if (!hp) return ATTN_ERR_CUDA;
    HostChunk ch[kHostChunks];
    const int n = host_chunks(p, ch);
    const size_t qrow = (size_t)p.M * p.D * 2, krow = (size_t)p.N * p.D * 2;  // bytes per head
    // the copies into q_d, k_d, v_d wait for the work already queued on the stream
    if (cudaEventRecord(hp->start, s) != cudaSuccess || cudaStreamWaitEvent(hp->h2d, hp->start, 0) != cudaSuccess)
        return ATTN_ERR_CUDA;
    int rc = ATTN_OK;
    for (int c = 0; c < n && rc == ATTN_OK; ++c) {
        const HostChunk& x = ch[c];
        const size_t qoff = ((size_t)x.b0 * p.Hq + (size_t)x.g0 * p.G) * qrow;
        const size_t koff = ((size_t)x.b0 * p.Hkv + x.g0) * krow;
        const size_t qbytes = (size_t)x.nb * x.ng * p.G * qrow, kbytes = (size_t)x.nb * x.ng * krow;
        if (cudaMemcpyAsync(q_d + qoff, q_h + qoff, qbytes, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
            cudaMemcpyAsync(k_d + koff, k_h + koff, kbytes, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
            cudaMemcpyAsync(v_d + koff, v_h + koff, kbytes, cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
            cudaEventRecord(hp->in[c], hp->h2d) != cudaSuccess || cudaStreamWaitEvent(s, hp->in[c], 0) != cudaSuccess) {
            rc = ATTN_ERR_CUDA;
            break;
        }
        Problem sub;
        rc = validate(q_d + qoff, k_d + koff, v_d + koff, o_d + qoff, x.nb, x.ng * p.G, x.ng, p.M, p.N, p.D, p.causal,
                      p.window, p.scale, p.dtype, &sub);
        if (rc == ATTN_OK) rc = run(sub, q_d + qoff, k_d + koff, v_d + koff, o_d + qoff, path, nullptr, 0, s);
        if (rc != ATTN_OK) break;
        if (cudaEventRecord(hp->done[c], s) != cudaSuccess || cudaStreamWaitEvent(hp->d2h, hp->done[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(o_h + qoff, o_d + qoff, qbytes, cudaMemcpyDeviceToHost, hp->d2h) != cudaSuccess)
            rc = ATTN_ERR_CUDA;
    }
    // drain every stream the call used, whatever happened above
    const cudaError_t e1 = cudaStreamSynchronize(hp->h2d);
    const cudaError_t e2 = cudaStreamSynchronize(s);
    const cudaError_t e3 = cudaStreamSynchronize(hp->d2h);
    if (rc == ATTN_OK && (e1 != cudaSuccess || e2 != cudaSuccess || e3 != cudaSuccess)) rc = ATTN_ERR_CUDA;
    return rc;
}

}  // namespace

int validate_problem(const void* q, const void* k, const void* v, const void* o, int B, int Hq, int Hkv, int M,
                     int N, int D, int causal, int window, float scale, int dtype, Problem* p) {
    return validate(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, p);
}

int* device_status_ptr() { return status_ptr(); }

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const cudaError_t e = once_per_device(g_sm_once, [dev] {
        return cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    });
    return e == cudaSuccess ? g_sm_count[dev] : 0;
}

size_t split_workspace_bytes(int rows, int S, int D) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t ml = up((size_t)rows * S * sizeof(float));
    return 2 * ml + up((size_t)rows * S * D * sizeof(float));
}

SplitWorkspace split_workspace(void* base, int rows, int S, int D) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t ml = up((size_t)rows * S * sizeof(float));
    (void)D;
    char* c = static_cast<char*>(base);
    return SplitWorkspace{reinterpret_cast<float*>(c), reinterpret_cast<float*>(c + ml),
                          reinterpret_cast<float*>(c + 2 * ml)};
}

}  // namespace attn

using namespace attn;

extern "C" {

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int M, int N, int D,
                int causal, int window, float scale, attn_dtype_t dtype, int path, void* workspace, size_t ws_bytes,
                void* stream) {
    if (path < ATTN_PATH_AUTO || path > ATTN_PATH_PREFILL_PAIR) return ATTN_ERR_PATH;
    Problem p;
    int rc = validate(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    return run(p, q, k, v, o, choose_path(p, path), workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int M, int N, int D,
             int causal, int window, float scale, attn_dtype_t dtype, void* stream) {
    Problem p;
    int rc = validate(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    const int path = choose_path(p, ATTN_PATH_AUTO);
    const size_t bytes = empty_output(p) || p.N == 0 ? 0 : workspace_for(p, path);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (bytes == 0) return run(p, q, k, v, o, path, nullptr, 0, s);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = run(p, q, k, v, o, path, ws, bytes, s);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}

int attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int M,
                 int N, int D, int causal, int window, float scale, attn_dtype_t dtype, int path, void* workspace,
                 size_t ws_bytes, void* stream) {
    if (path < ATTN_PATH_AUTO || path > ATTN_PATH_PREFILL_PAIR) return ATTN_ERR_PATH;
    Problem p;
    int rc = validate(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    if (!empty_output(p) && !lse) return ATTN_ERR_NULL;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_ERR_ALIGN;
    p.lse = lse;
    path = choose_path(p, path);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = empty_output(p) || p.N == 0 ? 0 : workspace_for(p, path);
    if (workspace || bytes == 0) return run(p, q, k, v, o, path, workspace, ws_bytes, s);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = run(p, q, k, v, o, path, ws, bytes, s);
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}

size_t attn_workspace_bytes_ex(int B, int Hq, int Hkv, int M, int N, int D, int causal, int window, int path) {
    Problem p;
    // placeholder non-null pointers: only the shape is checked here
    static const int16_t dummy[8] __attribute__((aligned(16))) = {};
    if (validate(dummy, dummy, dummy, dummy, B, Hq, Hkv, M, N, D, causal, window, 0.f, ATTN_BF16, &p) != ATTN_OK)
        return 0;
    if (path < ATTN_PATH_AUTO || path > ATTN_PATH_PREFILL_PAIR) return 0;
    if (empty_output(p) || p.N == 0) return 0;
    return workspace_for(p, choose_path(p, path));
}

size_t attn_workspace_bytes(int B, int Hq, int Hkv, int M, int N, int D, int window) {
    const size_t a = attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, 0, window, ATTN_PATH_AUTO);
    const size_t b = attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, 1, window, ATTN_PATH_AUTO);
    return a > b ? a : b;
}

int attn_fwd_ws(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv, int M, int N, int D,
                int causal, int window, float scale, attn_dtype_t dtype, void* workspace, size_t ws_bytes,
                void* stream) {
    Problem p;
    int rc = validate(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    const int path = choose_path(p, ATTN_PATH_AUTO);
    // the caller's workspace is checked before anything is launched
    const size_t need = empty_output(p) || p.N == 0 ? 0 : workspace_for(p, path);
    if (need > 0 && (!workspace || ws_bytes < need)) return ATTN_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return ATTN_ERR_ALIGN;
    return run(p, q, k, v, o, path, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int attn_merge(const float* m, const float* l, const float* acc, void* o, float* m_out, float* l_out, int rows,
               int S, int D, attn_dtype_t out_dtype, void* stream) {
    if (rows < 0 || S < 1 || S > 4096 || D < 1 || D > 256) return ATTN_ERR_SHAPE;
    if (out_dtype != ATTN_BF16 && out_dtype != ATTN_FP16 && out_dtype != ATTN_FP32) return ATTN_ERR_DTYPE;
    if ((int64_t)rows * S * D > kI32Max) return ATTN_ERR_OVERFLOW;
    if (rows == 0) return ATTN_OK;
    if (!m || !l || !acc || !o) return ATTN_ERR_NULL;
    return cuda_status(launch_merge(m, l, acc, o, m_out, l_out, nullptr, rows, S, D, out_dtype, kLog2e, false,
                                    static_cast<cudaStream_t>(stream)));
}

int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, void* q_d, void* k_d, void* v_d,
                  void* o_d, int B, int Hq, int Hkv, int M, int N, int D, int causal, int window, float scale,
                  attn_dtype_t dtype, void* workspace, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = validate(q_d, k_d, v_d, o_d, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    const size_t qb = (size_t)B * Hq * M * D * 2, kb = (size_t)B * Hkv * N * D * 2;
    if ((qb && (!q_h || !o_h)) || (kb && (!k_h || !v_h))) return ATTN_ERR_NULL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int path = choose_path(p, ATTN_PATH_AUTO);
    // prefill and SIMT problems need no workspace, so their chunks run as
    // independent problems with copies overlapping compute
    if (path != ATTN_PATH_DECODE && qb > 0 && kb > 0 && p.B * p.Hkv > 1)
        return run_host_pipelined(p, static_cast<const char*>(q_h), static_cast<const char*>(k_h),
                                  static_cast<const char*>(v_h), static_cast<char*>(o_h), static_cast<char*>(q_d),
                                  static_cast<char*>(k_d), static_cast<char*>(v_d), static_cast<char*>(o_d), path, s);
    if (qb && cudaMemcpyAsync(q_d, q_h, qb, cudaMemcpyHostToDevice, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (kb && cudaMemcpyAsync(k_d, k_h, kb, cudaMemcpyHostToDevice, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (kb && cudaMemcpyAsync(v_d, v_h, kb, cudaMemcpyHostToDevice, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = run(p, q_d, k_d, v_d, o_d, path, workspace, ws_bytes, s);
    if (rc != ATTN_OK) return rc;
    if (qb && cudaMemcpyAsync(o_h, o_d, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(s));
}

const char* attn_strerror(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "a required pointer is NULL";
        case ATTN_ERR_SHAPE: return "invalid shape (negative size, or Hkv == 0 with Hq > 0)";
        case ATTN_ERR_DTYPE: return "unsupported dtype";
        case ATTN_ERR_HEADDIM: return "unsupported head dimension for this path";
        case ATTN_ERR_GQA: return "Hq is not a multiple of Hkv";
        case ATTN_ERR_OVERFLOW: return "element count exceeds signed 32-bit indexing";
        case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA call failed";
        case ATTN_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
        case ATTN_ERR_PATH: return "the requested path cannot run this problem";
        default: return "unknown status";
    }
}

int attn_last_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    return word ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

int attn_version(void) { return 200; }

}  // extern "C"

extern "C" {

size_t attn_bwd_workspace_bytes(int B, int Hq, int M) {
    if (B < 0 || Hq < 0 || M < 0) return 0;
    if ((int64_t)B * Hq * M == 0) return 0;
    return bwd_workspace_bytes(B, Hq, M);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o, const float* lse, void* dq,
             void* dk, void* dv, int B, int Hq, int Hkv, int M, int N, int D, int causal, int window, float scale,
             attn_dtype_t dtype, void* workspace, size_t ws_bytes, void* stream) {
    Problem p;
    int rc = validate(q, k, v, o, B, Hq, Hkv, M, N, D, causal, window, scale, dtype, &p);
    if (rc != ATTN_OK) return rc;
    if (D != 16 && D != 32 && D != 64 && D != 128) return ATTN_ERR_HEADDIM;
    // the CUDA-core kernels of D = 16, 32 take one (batch, head) per grid y index
    if (D < 64 && (int64_t)B * Hq > 65535) return ATTN_ERR_PATH;
    const int64_t nq = (int64_t)B * Hq * M * D, nk = (int64_t)B * Hkv * N * D;
    if ((nq > 0 && (!d_o || !lse || !dq)) || (nk > 0 && (!dk || !dv))) return ATTN_ERR_NULL;
    if ((d_o && !aligned16(d_o)) || (dq && !aligned16(dq)) || (dk && !aligned16(dk)) || (dv && !aligned16(dv)) ||
        (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
        return ATTN_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // no query row, or no key: the gradients that exist are zero
    if (nq == 0 || nk == 0) {
        if (nq > 0 && cudaMemsetAsync(dq, 0, (size_t)nq * 2, s) != cudaSuccess) return ATTN_ERR_CUDA;
        if (nk > 0 && (cudaMemsetAsync(dk, 0, (size_t)nk * 2, s) != cudaSuccess ||
                       cudaMemsetAsync(dv, 0, (size_t)nk * 2, s) != cudaSuccess))
            return ATTN_ERR_CUDA;
        return ATTN_OK;
    }
    int* status = status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    BwdArgs a{q, k, v, o, d_o, lse, dq, dk, dv};
    const size_t need = bwd_workspace_bytes(B, Hq, M);
    if (workspace) {
        if (ws_bytes < need) return ATTN_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
        return cuda_status(launch_bwd(p, a, workspace, status, s));
    }
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return ATTN_ERR_CUDA;
    rc = cuda_status(launch_bwd(p, a, ws, status, s));
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}

}  // extern "C"

extern "C" {

size_t attn_split_softmax_workspace_bytes(int M, int N, int chunk) {
    if (M < 0 || M > 65535 || N < 1 || N > 131072 || !split_softmax_chunk_ok(chunk)) return 0;
    return split_softmax_ws_bytes(M, N, chunk);
}

int attn_split_softmax(const void* x, void* y, int M, int N, int chunk, attn_dtype_t dtype, void* workspace, size_t ws_bytes,
                       void* stream) {
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16 && dtype != ATTN_FP32) return ATTN_ERR_DTYPE;
    if (M < 0 || M > 65535 || N < 1 || N > 131072 || !split_softmax_chunk_ok(chunk)) return ATTN_ERR_SHAPE;
    if ((int64_t)M * N > kI32Max) return ATTN_ERR_OVERFLOW;
    if (M == 0) return ATTN_OK;
    if (!x || !y) return ATTN_ERR_NULL;
    if (!aligned16(x) || !aligned16(y)) return ATTN_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t need = split_softmax_ws_bytes(M, N, chunk);
    if (need == 0) return cuda_status(launch_split_softmax(x, y, M, N, chunk, dtype, nullptr, s));
    if (workspace) {
        if (ws_bytes < need) return ATTN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 7u) return ATTN_ERR_ALIGN;
        return cuda_status(launch_split_softmax(x, y, M, N, chunk, dtype, workspace, s));
    }
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, need, s) != cudaSuccess) return ATTN_ERR_CUDA;
    int rc = cuda_status(launch_split_softmax(x, y, M, N, chunk, dtype, ws, s));
    if (cudaFreeAsync(ws, s) != cudaSuccess && rc == ATTN_OK) rc = ATTN_ERR_CUDA;
    return rc;
}

}  // extern "C"
