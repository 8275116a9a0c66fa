// Self-tests of the failure-reporting path. attn_selftest_bounded_wait: one CTA
// waits on an mbarrier phase that nothing completes, with the same bounded-wait
// pattern the kernels use (poll, then give up after a time limit), and reports
// through the device status word. attn_selftest_prefill_abort: the real prefill
// kernel with one P-ready arrival withheld, so its issuing warp's wait runs out
// and every CTA takes its abort path (drain copies and MMAs, free TMEM, exit).
// Nothing faults, traps or hangs: the kernels return normally.
#include "attn_internal.h"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

__global__ void attn_selftest_wait_kernel(int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(b, 0)) {  // nobody arrives: phase 0 never completes
            if (globaltimer_ns() - t0 > limit_ns) {
                atomicExch(status, 1);
                break;
            }
        }
        mbar_arrive(b);  // leave the barrier's phase complete before the CTA exits
    }
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_selftest_bounded_wait(unsigned timeout_us, void* stream) {
    if (timeout_us == 0 || timeout_us > 2000000u) return ATTN_ERR_SHAPE;
    int* status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    attn_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, 1000ull * timeout_us);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

extern "C" int attn_selftest_prefill_abort(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                                           int Hkv, int M, int N, int D, attn_dtype_t dtype, long long withhold_at,
                                           void* stream) {
    Problem p;
    int rc = validate_problem(q, k, v, o, B, Hq, Hkv, M, N, D, 0, 0, 0.f, dtype, &p);
    if (rc != ATTN_OK) return rc;
    if (D != 128) return ATTN_ERR_HEADDIM;
    if ((int64_t)B * Hq * M == 0 || N == 0 || withhold_at < 0) return ATTN_ERR_SHAPE;
    if (!prefill_supported(p)) return ATTN_ERR_PATH;
    int* status = device_status_ptr();
    if (!status) return ATTN_ERR_CUDA;
    return launch_prefill_withheld(p, q, k, v, o, status, (long)withhold_at, static_cast<cudaStream_t>(stream));
}
