// Self-test of the bounded pipeline wait (sm_103a).
//
// Every mbarrier wait in the attention kernels gives up after a fixed time,
// raises ATTN_SINK_DEV_TIMEOUT and lets its kernel drain and return, so that a
// stalled pipeline becomes a status the host reads instead of a GPU that no
// longer answers.  This single-thread kernel runs that same wait (mbar_wait) on
// a barrier of its own.  With `complete` set it first completes the barrier's
// phase, so the wait returns at once; otherwise nothing ever arrives, the wait
// reaches its time limit, raises the status bit and the kernel returns.
#include "common.cuh"
#include "selftest.h"
#include "sm103.cuh"

namespace attn {
namespace selftest {

using namespace sm103;

__global__ void __launch_bounds__(1) wait_kernel(int complete) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (complete) mbar_arrive(&bar);
    mbar_wait(&bar, 0, &abort_flag);  // false (and the status bit) after the limit
}

cudaError_t launch_wait(int complete, cudaStream_t s) {
    wait_kernel<<<1, 1, 0, s>>>(complete ? 1 : 0);
    return cudaGetLastError();
}

ATTN_DEFINE_STATUS_ACCESSOR(status_exchange)

}  // namespace selftest
}  // namespace attn
