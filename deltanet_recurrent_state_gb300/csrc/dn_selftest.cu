// dn_wait_selftest: the bounded waits that the prefill kernels use, checked on the device
// without a fault, with the same functions the kernels call.
//  1. On an mbarrier that nothing arrives on, the guarded wait gives up once its time budget
//     has passed, raises the CTA's abort flag and counts the failure once.
//  2. After the one expected arrival, the same wait returns.
//  3. The drain path: a real bulk copy (global -> shared) is in flight when a second wait runs
//     out and raises the abort flag; the drain then waits (bounded) for that copy, which lands
//     with the bytes it was given.
// Nothing here waits without a bound, and no copy or address is invalid.
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_internal.h"
#include "dn_mma.cuh"

namespace dn {
namespace {

__global__ void wait_selftest_kernel(int budget_us, int32_t *result) {
    __shared__ __align__(16) int32_t landed[4];
    __shared__ __align__(8) unsigned long long mb[3];
    __shared__ int abort_flag;
    __shared__ unsigned int timeouts;
    const unsigned long long budget = (unsigned long long)budget_us * 1000ull;
    int32_t before[4];
    for (int i = 0; i < 4; ++i) before[i] = result[i];  // the bytes the copy of step 3 carries
    if (threadIdx.x == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&mb[i], 1);  // one arrival completes phase 0
        abort_flag = 0;
        timeouts = 0u;
        for (int i = 0; i < 4; ++i) landed[i] = 0;
        fence_proxy_async();
    }
    __syncthreads();
    // 1. nothing arrives on mb[0]: the wait runs out
    const bool done_early = mbar_wait_guarded(&mb[0], 0u, &abort_flag, &timeouts, budget);
    __syncthreads();
    const bool raised = abort_flag != 0;
    __syncthreads();
    // 2. with the flag lowered again and the arrival made, the wait on mb[1] returns
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_arrive_expect_tx(&mb[1], 0u);  // the arrival (no bytes announced)
    }
    __syncthreads();
    const bool done_late = mbar_wait_guarded(&mb[1], 0u, &abort_flag, &timeouts, budget);
    __syncthreads();
    // 3. a copy in flight when the CTA aborts: issue it, let a wait run out, then drain it
    bool drained = false;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&mb[2], 16u);
        bulk_load(landed, result, 16u, &mb[2]);
        const bool second = mbar_wait_guarded(&mb[0], 0u, &abort_flag, &timeouts, budget);  // runs out
        drained = !second && abort_flag != 0 && mbar_drain(&mb[2], 0u, budget);
        for (int i = 0; i < 4; ++i) drained = drained && landed[i] == before[i];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        result[0] = (!done_early && raised) ? 1 : 0;  // 1: the unfinished wait gave up and raised the flag
        result[1] = done_late ? 1 : 0;                // 1: the finished wait returned
        result[2] = drained ? 1 : 0;                  // 1: the copy in flight was drained and landed
        result[3] = (int32_t)timeouts;                // 2: each CTA-level failure counted once
    }
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_wait_selftest(int budget_us, int32_t *result, dn_stream_t stream) {
    using namespace dn;
    if (budget_us < 1 || budget_us > 1000000 || !result || !aligned(result, 16)) return DN_ERR_INVALID_ARG;
    wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(budget_us, result);
    return launch_status();
}
