// Test-only kernel that makes the library's bounded mbarrier waits run out.
//
// It is built apart from librs with a short limit (-DRS_WAIT_LIMIT_NS) and
// waits, through the library's own mbar_wait and wait_or_abort, on an
// mbarrier that no thread ever arrives at.  Each wait must give up after the
// limit; wait_or_abort must also raise the abort flag and RS_DEV_TIMEOUT in
// the status word, and a later wait must see the flag and return at once.
// Nothing faults and nothing hangs: every wait is bounded by %globaltimer.
#include "rs_plan.cuh"

namespace {

__global__ void wait_timeout_kernel(uint32_t *status, unsigned long long *ns, int *res) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        rs::mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const unsigned long long t0 = rs::global_ns();
    const bool w1 = rs::mbar_wait(&bar, 0);
    const unsigned long long t1 = rs::global_ns();
    const bool w2 = rs::wait_or_abort(&bar, 0, &abort_flag, status);
    const unsigned long long t2 = rs::global_ns();
    __syncthreads();  // every thread has given up; the flag is raised
    const bool w3 = rs::wait_or_abort(&bar, 0, &abort_flag, status);
    const unsigned long long t3 = rs::global_ns();
    if (threadIdx.x == 0) {
        res[0] = w1; res[1] = w2; res[2] = w3; res[3] = abort_flag;
        ns[0] = t1 - t0; ns[1] = t2 - t1; ns[2] = t3 - t2; ns[3] = rs::kWaitLimitNs;
    }
}

}  // namespace

// status: device [1]; ns: device [4] (the three waits' durations and the
// limit); res: device [4] (the three waits' results and the abort flag).
extern "C" int rs_test_wait_timeout(uint32_t *status, unsigned long long *ns, int *res, void *stream) {
    wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(status, ns, res);
    return (int)cudaGetLastError();
}
