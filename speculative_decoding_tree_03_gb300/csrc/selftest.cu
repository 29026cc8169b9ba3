// selftest.cu -- a wait that runs out, on purpose.
//
// Every wait of the library's kernels on an mbarrier is bounded: after its
// deadline the waiting CTA raises its abort flag, leaves its loops, releases
// what it holds and reports SVF_DEV_TIMEOUT in the caller's status array, so
// the context stays usable. This kernel drives that path without any fault:
// it waits, with the same helpers and a short caller-chosen deadline, on an
// mbarrier that nothing ever arrives at, in one CTA and in a cluster of two
// CTAs (the distributed-shared-memory wait of the acceptance walk).
#include "common.cuh"
#include "internal.h"

namespace svf {

namespace {

// result[0]: CTA wait status, result[1]: its elapsed microseconds;
// result[2] / result[3]: the same for the cluster wait (rank 0 reports).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32)
    selftest_wait_kernel(int32_t *__restrict__ result, unsigned long long deadline_ns) {
    __shared__ uint64_t bar[2];
    __shared__ int abort_flag;
    const unsigned rank = blockIdx.x & 1u;
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    cluster_arrive();
    cluster_wait();
    if (threadIdx.x == 0) {
        // a CTA-local barrier nobody arrives at
        unsigned long long t0 = globaltimer_ns();
        const bool ok = mbar_wait_for(&bar[0], 0, &abort_flag, deadline_ns);
        unsigned long long t1 = globaltimer_ns();
        if (rank == 0) {
            result[0] = ok ? 0 : SVF_DEV_TIMEOUT;
            result[1] = (int32_t)((t1 - t0) / 1000ull);
        }
        // a barrier whose completion would come from the peer CTA, which
        // never sends it
        t0 = globaltimer_ns();
        const bool okc = mbar_wait_cluster_for(&bar[1], 0, deadline_ns);
        t1 = globaltimer_ns();
        if (rank == 0) {
            result[2] = okc ? 0 : SVF_DEV_TIMEOUT;
            result[3] = (int32_t)((t1 - t0) / 1000ull);
        }
    }
    __syncthreads();
    // neither CTA leaves while the other could still address its memory
    cluster_arrive();
    cluster_wait();
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t *result, unsigned long long deadline_ns,
                                 cudaStream_t stream) {
    selftest_wait_kernel<<<2, 32, 0, stream>>>(result, deadline_ns);
    return cudaGetLastError();
}

}  // namespace svf
