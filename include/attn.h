/*
 * attn.h -- C ABI of the GB300 (sm_103a) streaming attention forward library.
 *
 * The operation (every entry point below computes it or one of its parts):
 *   O[b,h,i,:] = sum_j softmax_j(scale * <Q[b,h,i,:], K[b,g,j,:]>) V[b,g,j,:]
 * over the keys j that row i may see, computed as a stream over key tiles that
 * carries a running (m, l, acc) state per row and never forms the full score
 * matrix ("Intermediate and advanced kernel workshops", table "Scope and
 * contracts", streaming_attention.attention row; answer key, central-idea
 * table, A3 row: each row keeps a running (m, l, a), and only one tile of scores
 * exists at any time).
 *
 * Conventions shared by every entry point:
 *   Layout      Q and O are [B, Hq, M, D]; K and V are [B, Hkv, N, D]; all
 *               row-major and contiguous, D innermost. The pages define one
 *               head [N, D] contiguous; batching and heads are this library's
 *               extension.
 *   GQA         query head h reads KV head g = h / (Hq / Hkv); Hq % Hkv == 0.
 *   Positions   query row i sits at key position p_i = i + N - M
 *               (bottom-right alignment; with M == N it is the pages' rule).
 *   causal      != 0 keeps keys j <= p_i (a row sees its own position).
 *   window      W > 0 keeps keys j > p_i - W (the W keys ending at p_i);
 *               W <= 0 disables it.
 *   scale       multiplies the logits; 0.0f selects the pages' 1/sqrt(D).
 *   Masked keys score -inf ("Kernel Notes & Checklist", gotchas ledger:
 *               masked and padded columns must be -inf, never 0). A row with
 *               no visible key (N == 0, or causal with p_i < 0) outputs 0,
 *               never NaN (same ledger, ghost rows).
 *   Precision   FP16 or BF16 in and out, FP32 accumulation, one cast at the
 *               end (scope table: FP32 epilogue, then one output cast). P is
 *               rounded to the input type before the P.V product (contract
 *               notes under the scope table). attn_fwd_fp8 and
 *               attn_decode_paged_fp8 take E4M3 inputs instead (see there).
 *   dtype       every dtype / out_dtype argument is an attn_dtype_t (an
 *               int-sized enum): ATTN_BF16 or ATTN_FP16, and ATTN_FP32 where an
 *               entry point says so.
 *   Pointers    q, k, v, o are DEVICE pointers owned by the caller, 16-byte
 *               aligned; o must not overlap q, k or v. They may be NULL only
 *               when the tensor has zero elements.
 *   Streams     `stream` is a cudaStream_t passed as void* so that this header
 *               needs no CUDA header (NULL = legacy default stream).
 *               Every call is asynchronous on it and never synchronizes,
 *               except attn_fwd_host and attn_last_device_status.
 *   Devices     calls run on the current CUDA device. Per-device setup (kernel
 *               shared-memory limits, the SM count, the status word's address)
 *               happens on the first call with that device current, so one
 *               process may drive several GPUs.
 *   Values      only metadata is validated, never values (scope notes: wrappers
 *               validate metadata but do not scan values); inputs must be
 *               finite. Every tensor's element count must fit a signed 32-bit
 *               index (same notes).
 *   Errors      a negative attn_status_t; nothing is thrown across the ABI.
 *               On a validation error no kernel has been launched.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

/* Exported symbols stay visible when the library is built with hidden default visibility. */
#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1, ATTN_FP32 = 2 } attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,      /* a required pointer is NULL */
    ATTN_ERR_SHAPE = -2,     /* a negative size, or Hkv == 0 with Hq > 0 */
    ATTN_ERR_DTYPE = -3,     /* dtype is not ATTN_BF16 / ATTN_FP16 */
    ATTN_ERR_HEADDIM = -4,   /* D is not supported by the requested path */
    ATTN_ERR_GQA = -5,       /* Hq is not a multiple of Hkv */
    ATTN_ERR_OVERFLOW = -6,  /* an element count does not fit a signed 32-bit index */
    ATTN_ERR_ALIGN = -7,     /* a pointer is not 16-byte aligned */
    ATTN_ERR_WORKSPACE = -8, /* workspace NULL or smaller than the size query returns */
    ATTN_ERR_CUDA = -9,      /* a CUDA runtime/driver call failed (launch, copy, ...) */
    ATTN_ERR_TIMEOUT = -10,  /* a kernel gave up on a bounded wait (see attn_last_device_status) */
    ATTN_ERR_PATH = -11      /* the requested path cannot run this problem */
} attn_status_t;

/* Kernel paths. AUTO picks: split-KV decode when (Hq/Hkv)*M <= 16 and the
 * visible key range is long; the tcgen05 prefill kernel for D in {64, 128};
 * the SIMT kernel otherwise (D in {16, 32, 64, 128}).
 * The SIMT kernel, which also runs split decode for B*Hkv > 65535 and the
 * log-sum-exp of an N == 0 call,
 * takes at most 65535 (batch, query head) pairs: B*Hq > 65535 there returns
 * ATTN_ERR_PATH (AUTO then prefers the prefill kernel for D in {64, 128}). */
typedef enum {
    ATTN_PATH_AUTO = 0,
    ATTN_PATH_SIMT = 1,    /* CUDA-core streaming kernel, any supported D, B*Hq <= 65535 */
    ATTN_PATH_PREFILL = 2, /* warp-specialized TMA + tcgen05 + TMEM kernel, D in {64,128} */
    ATTN_PATH_DECODE = 3,  /* split-KV over grouped query heads (tcgen05, D = 64 or 128: the grouped
                              rows of a KV head in CTAs of 16); the splits merged in a thread-block
                              cluster (at most 8 splits per KV head) or by the merge kernel */
    ATTN_PATH_PREFILL_PAIR = 4 /* the prefill on the pair MMA (tcgen05 cta_group::2): clusters of two
                              CTAs share 512-row work tiles, each loading half of every K/V tile;
                              D = 128, BF16/FP16; never chosen by AUTO */
} attn_path_t;

/* Forward attention, the library's main entry point.
 *   q [B,Hq,M,D], k/v [B,Hkv,N,D], o [B,Hq,M,D]: device pointers (see above).
 *   dtype: ATTN_BF16 or ATTN_FP16 for all four tensors.
 * Picks the path as ATTN_PATH_AUTO does. When that path needs workspace
 * (split-KV decode) it is allocated stream-ordered on `stream` with
 * cudaMallocAsync and released with cudaFreeAsync after the launches.
 * Empty problems: B*Hq == 0 or M == 0 launches nothing; N == 0 zero-fills o.
 * Returns ATTN_OK or a negative status. */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o,
                      int B, int Hq, int Hkv, int M, int N, int D,
                      int causal, int window, float scale, attn_dtype_t dtype, void* stream);

/* Per-call scratch. The split-KV decode path keeps one partial summary
 * (m, l, acc[D]) per (query row, split) in device scratch that lives for one
 * call, the same arrangement as the course's wide-row split softmax
 * ("Intermediate and advanced kernel workshops", level table, A2: three
 * ordered kernels with per-call scratch; answer key, worked answer A2, where
 * 4 rows x 33 chunks need 1088 scratch bytes). The caller may own that scratch
 * (attn_fwd_ws, attn_fwd_ex) instead of having attn_fwd allocate it.
 * Layout: three 256-byte-aligned parts, m[rows][S] and l[rows][S] (float,
 * m in base-2 logit units) and acc[rows][S][D] (float), rows = B*Hq*M, S the
 * number of splits the library plans for the problem. */

/* Bytes of workspace attn_fwd_ws needs for a problem of these sizes (the path
 * attn_fwd would take), enough for either value of `causal`; 0 when that path
 * needs none, for empty problems and for invalid shapes. */
ATTN_API size_t attn_workspace_bytes(int B, int Hq, int Hkv, int M, int N, int D, int window);

/* attn_fwd with caller-owned device workspace instead of a stream-ordered
 * allocation: the same path choice (ATTN_PATH_AUTO) and the same result.
 *   workspace: device memory of at least attn_workspace_bytes(B, Hq, Hkv, M,
 *         N, D, window) bytes, 16-byte aligned; NULL (with ws_bytes 0) is
 *         allowed when that size is 0. A smaller or missing workspace on a
 *         path that needs one returns ATTN_ERR_WORKSPACE with nothing
 *         launched. The memory must stay untouched until the work queued on
 *         `stream` has finished; its contents need no clearing. */
ATTN_API int attn_fwd_ws(const void* q, const void* k, const void* v, void* o,
                         int B, int Hq, int Hkv, int M, int N, int D,
                         int causal, int window, float scale, attn_dtype_t dtype,
                         void* workspace, size_t ws_bytes, void* stream);

/* Bytes of caller workspace that attn_fwd_ex needs for this problem on this
 * path (0 when the path needs none). Returns 0 for invalid shapes too. */
ATTN_API size_t attn_workspace_bytes_ex(int B, int Hq, int Hkv, int M, int N, int D,
                                        int causal, int window, int path);

/* attn_fwd with an explicit path and caller-owned device workspace.
 *   path: an attn_path_t; a forced path that cannot run the problem returns
 *         ATTN_ERR_PATH (or ATTN_ERR_HEADDIM for an unsupported D).
 *   workspace: device memory of at least attn_workspace_bytes_ex(...) bytes
 *         for the same problem and path, 16-byte aligned, or NULL when that
 *         is 0. It must stay untouched until the work queued on `stream` has
 *         finished. */
ATTN_API int attn_fwd_ex(const void* q, const void* k, const void* v, void* o,
                         int B, int Hq, int Hkv, int M, int N, int D,
                         int causal, int window, float scale, attn_dtype_t dtype, int path,
                         void* workspace, size_t ws_bytes, void* stream);

/* attn_fwd_ex that also writes each row's log-sum-exp of its logits,
 *   lse[b,h,i] = ln sum_{j visible} exp(scale * <Q[b,h,i,:], K[b,g,j,:]>),
 * natural log, -inf for a row with no visible key: the summary (m, l) of the
 * answer key's A1 row folded into one number (m + ln l), which the backward
 * pass needs and with which the outputs of calls over disjoint key ranges merge
 * (attn_merge with m = lse, l = 1, acc = o).
 *   lse: device float [B, Hq, M], 4-byte aligned, owned by the caller; NULL only
 *        when the output is empty.
 *   workspace: as attn_fwd_ex, or NULL to have it allocated stream-ordered
 *        (cudaMallocAsync / cudaFreeAsync) as attn_fwd does. */
ATTN_API int attn_fwd_lse(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int M, int N, int D,
                          int causal, int window, float scale, attn_dtype_t dtype, int path,
                          void* workspace, size_t ws_bytes, void* stream);

/* Forward pass on 8-bit E4M3 inputs (the OCP 8-bit floating-point E4M3
 * encoding: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals,
 * no infinities, S.1111.111 is NaN) with per-tensor dequantization factors:
 * the operation is the forward pass of attn_fwd on the dequantized tensors
 *   Q = q_descale * q, K = k_descale * k, V = v_descale * v,
 *   O = softmax(scale * Q K^T over the visible keys) V,
 * written as BF16 or FP16 (out_dtype). Both products run on the tensor cores
 * with 8-bit operands: the probabilities P (relative to each row's running
 * reference maximum, at most 2^8) are rounded to E4M3 before the value
 * product, while the row sum l adds the unrounded FP32 values. The rounding
 * of P is the one approximation beyond FP32 accumulation: each output
 * element's error is at most 2^-4 times the weighted mean of |V| over its row
 * (plus 2^-10 / l per key for probabilities below E4M3's normal range).
 * An FP8 extension of the tcgen05 kernels: the pages use 16-bit inputs only.
 *   q: device bytes [B, Hq, M, D]; k, v: device bytes [B, Hkv, N, D]; o: device
 *   [B, Hq, M, D] of out_dtype (ATTN_BF16 / ATTN_FP16, else ATTN_ERR_DTYPE); all
 *   16-byte aligned. lse: as attn_fwd_lse (of the dequantized logits), or NULL.
 *   D is 128 or 64 (else ATTN_ERR_HEADDIM); D = 64 runs the prefill kernel's
 *   128-column form with the upper 64 columns of every tile read as zeros.
 *   Descale factors must be finite (not checked).
 *   path: ATTN_PATH_AUTO (split-KV decode when D = 128, (Hq/Hkv) * M <= 16 and
 *   the visible key range spans at least 512 keys, else prefill),
 *   ATTN_PATH_PREFILL, or ATTN_PATH_DECODE (D = 128 only, any number of grouped
 *   rows, in CTAs of 16); ATTN_PATH_SIMT is not offered (ATTN_ERR_PATH).
 *   workspace: for the decode path, attn_fwd_fp8_workspace_bytes(...) bytes of
 *   the same problem and path (the 8-bit kernel runs more splits than the
 *   16-bit one), 16-byte aligned, or NULL to have it allocated stream-ordered;
 *   the prefill path needs none.
 *   M == 0: nothing is written; N == 0: o is zero-filled (and lse set to -inf). */
/* Bytes of caller workspace attn_fwd_fp8 needs for this problem on this path
 * (0 for the prefill path, empty problems and invalid shapes). */
ATTN_API size_t attn_fwd_fp8_workspace_bytes(int B, int Hq, int Hkv, int M, int N, int D,
                                             int causal, int window, int path);
ATTN_API int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int M, int N, int D,
                          int causal, int window, float scale,
                          float q_descale, float k_descale, float v_descale,
                          attn_dtype_t out_dtype, int path, void* workspace, size_t ws_bytes, void* stream);

/* Backward pass: gradients of L = sum(dO * O) for O = attention(Q, K, V).
 * Each row of the weight gradient is the softmax vector-Jacobian product of
 * that row ("Intermediate and advanced kernel workshops", workshop I2, softmax
 * backward; answer key, I2 row and worked answer), with P recomputed from the
 * forward's log-sum-exp (attn_fwd_lse) instead of being stored:
 *   P = exp(scale Q K^T - lse) over the visible keys, dV = P^T dO,
 *   dP = dO V^T, dS = P * (dP - rowsum(dO * O)), dQ = scale dS K,
 *   dK = scale dS^T Q; with GQA, dK and dV of a KV head sum over its query heads.
 *   q, o, d_o, dq: device [B, Hq, M, D]; k, v, dk, dv: device [B, Hkv, N, D];
 *   all of dtype, 16-byte aligned; lse: device float [B, Hq, M] from the forward
 *   of the same q, k, v, causal, window and scale. dq, dk, dv are written (not
 *   accumulated) and must not overlap the inputs.
 *   D is 64 or 128 (tcgen05 kernels; P and dS rounded to dtype for their
 *   products) or 16 or 32 (CUDA-core kernels, P and dS kept in FP32, at most
 *   65535 (batch, query head) pairs, else ATTN_ERR_PATH); else ATTN_ERR_HEADDIM.
 *   M == 0 or N == 0: the gradients that exist are zero-filled.
 *   workspace: device memory of attn_bwd_workspace_bytes(B, Hq, M) bytes,
 *   16-byte aligned, or NULL to have it allocated stream-ordered. */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int Hq, int M);
ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* d_o,
                      const float* lse, void* dq, void* dk, void* dv,
                      int B, int Hq, int Hkv, int M, int N, int D,
                      int causal, int window, float scale, attn_dtype_t dtype,
                      void* workspace, size_t ws_bytes, void* stream);

/* Merge of split summaries, the pages' common-maximum rule (answer key,
 * central-idea table, A1 row, and its worked answer: (2,2) and (4,1) merge
 * to (4, 1+2e^-2)).
 *   m, l: device float [rows][S]; acc: device float [rows][S][D]. Summary s of
 *   a row is (m_s, l_s, acc_s) with l_s = sum exp(x - m_s) and acc_s the
 *   matching unnormalized sum of value rows; (-inf, 0, 0) is the empty one.
 *   o: device [rows][D] in out_dtype (ATTN_BF16, ATTN_FP16 or ATTN_FP32),
 *   receives sum_s w_s acc_s / sum_s w_s l_s with w_s = exp(m_s - max m), or
 *   0 when every summary is empty.
 *   m_out, l_out: optional device float [rows] (NULL to skip) receiving the
 *   merged summary.
 * rows >= 0, 1 <= S <= 4096, 1 <= D <= 256. */
ATTN_API int attn_merge(const float* m, const float* l, const float* acc, void* o,
                        float* m_out, float* l_out, int rows, int S, int D, attn_dtype_t out_dtype,
                        void* stream);

/* End-to-end call on HOST buffers: copies q, k, v from host memory into the
 * caller's device buffers, runs attn_fwd_ex with ATTN_PATH_AUTO, copies o back
 * to host memory, and synchronizes `stream` before returning. On the prefill
 * and SIMT paths the work is cut into up to 8 chunks of whole (batch, KV head)
 * groups whose copies run on two internal copy streams, overlapping the
 * kernels of other chunks on `stream` (the copies wait for the work already
 * queued on `stream`); the decode path copies, computes and copies back in
 * order on `stream`. Chunked calls from several host threads are serialized
 * (they share the internal copy streams and events).
 *   *_h: host pointers (pinned memory gives asynchronous copies);
 *   *_d: device buffers of the same sizes, owned by the caller;
 *   workspace/ws_bytes: as attn_fwd_ex (may be NULL/0 when none is needed).
 * Returns ATTN_OK, a validation status, or ATTN_ERR_CUDA. */
ATTN_API int attn_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                           void* q_d, void* k_d, void* v_d, void* o_d,
                           int B, int Hq, int Hkv, int M, int N, int D,
                           int causal, int window, float scale, attn_dtype_t dtype,
                           void* workspace, size_t ws_bytes, void* stream);

/* Split-KV decode forward that allocates no memory.
 * The source pages have no counterpart to this entry point: it exists for
 * callers that cannot allocate device memory when they run the forward --
 * for example code inside an allocator hook or custom memory pool (which must
 * not re-enter cudaMalloc), or a latency-critical loop whose rules forbid
 * allocation. attn_fwd would allocate the split workspace with
 * cudaMallocAsync, and attn_fwd_ex needs the caller to provide it.
 * Instead, this call keeps the split summaries in one fixed device array of
 * ATTN_NOALLOC_SCRATCH_BYTES bytes that the library holds on every GPU that
 * loads it, until the process exits. It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   Arguments, layout and errors are those of attn_fwd; the caller still
 *   provides q, k, v and o. D must be 64 or 128.
 *   Returns ATTN_ERR_WORKSPACE when the problem's split summaries
 *   (attn_workspace_bytes_ex(..., ATTN_PATH_DECODE)) exceed the array and the
 *   splits do not merge inside their cluster (see below), and
 *   ATTN_ERR_PATH when B*Hkv > 65535 and B*Hq > 65535 (the splits would run
 *   on the SIMT kernel, whose grid takes at most 65535 (batch, query head) pairs).
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   Every call, on any stream, shares the one array and leaves its contents
 *   behind: calls whose work may overlap on the GPU race and must be
 *   serialized by the caller (one stream, or events). Nothing in the array
 *   needs clearing: each call writes every summary it reads, including an
 *   empty one for a split that sees no key or gives up on a bounded wait (the
 *   output is then unspecified and attn_last_device_status reports it). When
 *   a KV head has at most 8 splits -- enough KV heads, as in
 *   typical GQA decode -- the splits merge inside their thread-block cluster,
 *   the array is not touched at all, and its size does not limit the problem. */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
ATTN_API int attn_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                     int B, int Hq, int Hkv, int M, int N, int D,
                                     int causal, int window, float scale, attn_dtype_t dtype, void* stream);

/* Split-KV decode over a PAGED KV cache: the KV-cache slice of the course's
 * plan ("Kernel Notes & Checklist", section 3, the plan, week +3: sliding
 * window + GQA + KV-cache slice). Each sequence b attends over its own first
 * L_b = min(seq_lens[b], max_pages * page_size, max_seq_len) keys, with the
 * conventions above (positions p_i = i + L_b - M, causal, window, GQA), so
 * the result equals attn_fwd on sequence b's keys gathered into a contiguous
 * [1, Hkv, L_b, D] cache.
 *   q, o        device [B, Hq, M, D], dtype, 16-byte aligned; M query rows per
 *               sequence (1 for decode, more for speculative decode).
 *   k_pages,    device pools [num_pages, Hkv, page_size, D], dtype, 16-byte
 *   v_pages     aligned: page n holds page_size consecutive keys of every KV
 *               head, each head's rows contiguous (the same head-major layout
 *               as k and v of attn_fwd). A contiguous [B, Hkv, Nmax, D] cache
 *               is the special case page_size = Nmax, max_pages = 1,
 *               block_table[b] = b.
 *   block_table device int32 [B, max_pages], 4-byte aligned: key j of
 *               sequence b is row j % page_size of page
 *               block_table[b * max_pages + j / page_size]. Only the entries
 *               of pages holding the first L_b keys are read; they must lie in
 *               [0, num_pages) (an entry outside reads a page of zeros: no
 *               fault, but a wrong result).
 *   seq_lens    device int32 [B], 4-byte aligned (negative counts as 0).
 *   page_size   16, 32, 64 or a multiple of 128.
 *   max_seq_len a host-side bound of the seq_lens values: it sizes the split
 *               plan; keys past it are ignored.
 *   D is 16, 32, 64 or 128 (else ATTN_ERR_HEADDIM); B * Hkv <= 65535 and at
 *   most 16 * 65535 (D = 64 and 128) or 8 * 65535 (D = 16 and 32) grouped
 *   rows (Hq/Hkv) * M per KV head (else ATTN_ERR_OVERFLOW).
 *   Kernels: D = 64 and 128 run the tcgen05 split kernel (pages gathered by
 *   TMA, the grouped rows of a KV head in CTAs of 16); D = 16 and 32 run a
 *   grouped CUDA-core kernel (one block per split, sequence, KV head and eight
 *   grouped rows, each 32-key tile gathered from its pages once for all of
 *   them). Both end in the same common-maximum merge.
 *   Every element of a page that a sequence uses must be finite, also in the
 *   rows of its last page past L_b: masked keys get probability 0, and their
 *   value rows are still multiplied by it.
 *   workspace: device memory of attn_decode_paged_workspace_bytes(...) bytes,
 *   16-byte aligned; NULL makes the call allocate it stream-ordered
 *   (cudaMallocAsync / cudaFreeAsync on `stream`), as attn_fwd does. The
 *   size is 0 when the grouped kernel plans one split per sequence (it then
 *   writes o itself) and the workspace is not read.
 *   When num_pages == 0 or min(max_seq_len, max_pages * page_size) == 0, o is
 *   zero-filled. */
ATTN_API size_t attn_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int M, int D,
                                                  int page_size, int max_pages, int max_seq_len,
                                                  int causal, int window);
ATTN_API int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                               const int* block_table, const int* seq_lens, void* o,
                               int B, int Hq, int Hkv, int M, int D,
                               int num_pages, int page_size, int max_pages, int max_seq_len,
                               int causal, int window, float scale, attn_dtype_t dtype,
                               void* workspace, size_t ws_bytes, void* stream);

/* attn_decode_paged on an E4M3 cache: q and both pools hold E4M3 bytes (the
 * encoding of attn_fwd_fp8) with per-tensor dequantization factors, and the
 * operation is attn_decode_paged of the dequantized tensors, written as
 * out_dtype (ATTN_BF16 / ATTN_FP16). The probabilities are rounded to E4M3
 * for the value product as in attn_fwd_fp8. Arguments and limits as
 * attn_decode_paged, except that D = 64 runs the grouped CUDA-core kernel (so
 * at most 8 * 65535 grouped rows); the workspace is attn_decode_paged_fp8_workspace_bytes(...)
 * bytes (or NULL to have it allocated stream-ordered). */
ATTN_API size_t attn_decode_paged_fp8_workspace_bytes(int B, int Hq, int Hkv, int M, int D,
                                                      int page_size, int max_pages,
                                                      int max_seq_len, int causal, int window);
ATTN_API int attn_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages,
                                   const int* block_table, const int* seq_lens, void* o,
                                   int B, int Hq, int Hkv, int M, int D, int num_pages,
                                   int page_size, int max_pages, int max_seq_len,
                                   int causal, int window, float scale,
                                   float q_descale, float k_descale, float v_descale, attn_dtype_t out_dtype,
                                   void* workspace, size_t ws_bytes, void* stream);

/* Wide-row split softmax, the course's workshop A2 ("Intermediate and advanced
 * kernel workshops": three ordered kernels with per-call scratch; answer key,
 * A2 row and worked answer): y[i,:] = softmax(x[i,:]) for each row of a
 * contiguous [M, N] matrix, computed as partial statistics per chunk of
 * `chunk` columns, their merge relative to the common maximum, then a reread
 * that normalizes, all on `stream`.
 *   x, y: device [M, N], dtype ATTN_FP32, ATTN_FP16 or ATTN_BF16 (both), 16-byte
 *         aligned; FP32 arithmetic, one cast of y. 1 <= N <= 131072; M >= 0
 *         (M == 0 launches nothing); M <= 65535.
 *   chunk: 256, 1024 or 4096 runs the three kernels with chunks of that many
 *         columns; 0 runs the row-resident form: the row's chunks (at most 8,
 *         of 4096 or 16384 columns) are the CTAs of one thread-block cluster,
 *         keep their values on chip, exchange their (max, sum) pairs through
 *         distributed shared memory, merge them the same way and normalize
 *         without rereading x (x read once, y written once).
 *   workspace: 8 * M * (ceil(N / chunk) + 1) bytes (a float pair per chunk and
 *         one merged pair per row), 8-byte aligned, or NULL to have it
 *         allocated stream-ordered; none for chunk 0 (workspace ignored).
 *         Values are not validated; x must be finite. */
ATTN_API size_t attn_split_softmax_workspace_bytes(int M, int N, int chunk);
ATTN_API int attn_split_softmax(const void* x, void* y, int M, int N, int chunk, attn_dtype_t dtype,
                                void* workspace, size_t ws_bytes, void* stream);

/* Human-readable text for a status code (static storage). */
ATTN_API const char* attn_strerror(int status);

/* Synchronizes `stream`, then returns and clears the device status word that
 * kernels set when a bounded wait gives up: ATTN_OK when none did, else
 * ATTN_ERR_TIMEOUT. ATTN_ERR_CUDA if the synchronization itself failed.
 * There is one status word per device, shared by every stream and host thread
 * that calls into the library on that device: a give-up on one stream is
 * reported to, and cleared by, whichever caller reads the word first (a caller
 * that needs per-stream attribution must serialize its status reads). */
ATTN_API int attn_last_device_status(void* stream);

/* Self-test of failure reporting: launches one CTA that waits on an mbarrier
 * phase nothing completes, gives up after timeout_us microseconds (1 ..
 * 2,000,000) exactly as the kernels' bounded waits do, and sets the device
 * status word; attn_last_device_status then returns ATTN_ERR_TIMEOUT. No fault,
 * trap or hang: the context stays usable. The pages have no counterpart. */
ATTN_API int attn_selftest_bounded_wait(unsigned timeout_us, void* stream);

/* Failure-path self-test of the prefill kernel itself: runs the noncausal
 * tcgen05 prefill (D = 128, dtype ATTN_BF16 / ATTN_FP16) on the caller's
 * device buffers (as attn_fwd) with the softmax warps of query tile 0
 * withholding their P-ready arrival at score tile `withhold_at` of each CTA's
 * walk. The issuing warp's bounded wait (1 s) runs out, and every CTA that
 * reaches that tile raises the abort flag, drains its copies and MMAs, frees
 * TMEM and exits; attn_last_device_status then returns ATTN_ERR_TIMEOUT and the
 * context stays usable. o is left unspecified. No fault, trap or hang.
 * Returns a validation status (withhold_at < 0 or an empty problem:
 * ATTN_ERR_SHAPE), ATTN_ERR_CUDA, or ATTN_OK once launched. */
ATTN_API int attn_selftest_prefill_abort(const void* q, const void* k, const void* v, void* o,
                                         int B, int Hq, int Hkv, int M, int N, int D, attn_dtype_t dtype,
                                         long long withhold_at, void* stream);

/* Library ABI version (major*100 + minor). 200: attn_workspace_bytes takes the
 * seven size arguments of attn_fwd_ws (the former nine-argument query is now
 * attn_workspace_bytes_ex), attn_fwd_ws is added, and dtype arguments are
 * typed attn_dtype_t (same size and values as before). 101 added the E4M3
 * entry points, chunk 0 of attn_split_softmax and attn_selftest_bounded_wait. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
