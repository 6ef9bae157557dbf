// dn_wait_selftest: the bounded wait that the prefill kernels use for their tensor-copy
// inputs, checked on the device in both directions. On an mbarrier that nothing arrives on,
// the wait has to give up after the given number of polls and say so (the kernels then count
// the failure instead of hanging); after the one expected arrival, the same wait has to
// succeed. Nothing here waits without a bound.
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_internal.h"
#include "dn_mma.cuh"

namespace dn {
namespace {

__global__ void wait_selftest_kernel(int tries, int32_t *result) {
    __shared__ unsigned long long mb;
    if (threadIdx.x == 0) mbar_init(&mb, 1);  // one arrival completes phase 0
    __syncthreads();
    const bool done_early = mbar_wait(&mb, 0u, tries);  // nothing has arrived: must run out
    __syncthreads();
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&mb, 0u);  // the arrival (no bytes announced)
    const bool done_late = mbar_wait(&mb, 0u, tries);    // phase 0 complete: must succeed
    if (threadIdx.x == 0) {
        result[0] = done_early ? 0 : 1;  // 1: the unfinished wait gave up
        result[1] = done_late ? 1 : 0;   // 1: the finished wait returned
    }
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_wait_selftest(int tries, int32_t *result, dn_stream_t stream) {
    using namespace dn;
    if (tries < 1 || tries > (1 << 20) || !result || !aligned(result, 4)) return DN_ERR_INVALID_ARG;
    wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(tries, result);
    return launch_status();
}
