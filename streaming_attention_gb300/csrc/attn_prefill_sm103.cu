#include "attn_internal.h"

namespace attn {

bool prefill_supported(const Problem& p) { (void)p; return false; }

int launch_prefill(const Problem& p, const void* q, const void* k, const void* v, void* o, int* status,
                   cudaStream_t stream) {
    (void)p; (void)q; (void)k; (void)v; (void)o; (void)status; (void)stream;
    return ATTN_ERR_PATH;
}

}  // namespace attn
