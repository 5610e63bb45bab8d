// Self-check of the bounded-wait give-up path shared by every kernel that
// waits on an mbarrier (the score, q.k and softmax value kernels).
//
// One CTA initialises an mbarrier that expects two arrivals, arrives once, and
// waits for the phase with the same bounded wait the kernels use, here with a
// caller-given limit.  The phase can never complete, so the wait gives up,
// records the timeout bit in this unit's status word and the kernel returns:
// nothing is copied and nothing else waits on it, so the context stays usable.
#include "common.cuh"

EKV_DEFINE_STATUS(selfcheck)

namespace ekv {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 2);
        mbar_fence_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        mbar_arrive(&bar);                 // the second arrival never comes
        if (!mbar_wait_for(&bar, 0, limit_ns)) flag_timeout();
    }
}

cudaError_t launch_wait_timeout_check(uint64_t limit_ns, cudaStream_t s) {
    return launch_kernel(wait_timeout_kernel, dim3(1), dim3(32), 0, s, limit_ns);
}

}  // namespace ekv
