// Self-test of the failure-reporting path: one CTA waits on an mbarrier phase
// that nothing completes, with the same bounded-wait pattern the kernels use
// (poll, then give up after a time limit), and reports through the device
// status word. Nothing faults, traps or hangs: the kernel returns normally.
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
