// Split-KV decode dispatch: the union key range [klo, khi) is cut into S
// chunks of whole 128-key tiles; each chunk's partial (m, l, acc) summaries
// go to the workspace, and the merge kernel combines them on the same stream
// ("Compare reasoning after your own attempt", central-idea table, A2 row:
// each split's statistics are combined after rescaling; the stream orders the kernels).
//
// D = 64 and 128 run the tcgen05 split kernel (grouped query rows in CTAs of
// 16); other shapes (B * Hkv > 65535) run the SIMT kernel in split mode.
#include "attn_internal.h"

namespace attn {

bool decode_supported(const Problem& p) { return p.D == 64 || p.D == 128; }

int decode_plan(const Problem& p, int* chunk, int* S) {
    if (decode_tc_supported(p)) return decode_plan_tc(p, chunk, S);
    const int kbase = split_base(p);
    const int range = p.khi > kbase ? p.khi - kbase : 1;
    int c = 256;
    int s = (range + c - 1) / c;
    if (s > 4096) {
        c = ((range + 4095) / 4096 + 127) / 128 * 128;
        s = (range + c - 1) / c;
    }
    *chunk = c;
    *S = s;
    return ATTN_OK;
}

cudaError_t launch_decode(const Problem& p, const void* q, const void* k, const void* v, int chunk, int S,
                          const SplitWorkspace& ws, int* status, cudaStream_t stream, DecodeOut* out) {
    if (decode_tc_supported(p)) return launch_decode_tc(p, q, k, v, chunk, S, ws, status, stream, out);
    if (out) out->merged = false;
    return launch_simt(p, q, k, v, nullptr, chunk, S, &ws, stream);
}

}  // namespace attn
