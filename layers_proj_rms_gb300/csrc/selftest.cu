// Self-test of the fault path: one thread waits, with the same bounded wait
// the tensor-core kernels use, on an mbarrier that nothing arrives at.  The
// wait runs out after `limit` SM clock cycles, the kernel reports
// kFaultSelfTest through the device fault word and returns, and the context
// stays usable.  Nothing faults, traps or hangs.
#include "launch.h"
#include "tc.cuh"

namespace mhc {

__global__ void k_selftest_wait(long long limit, int *fault)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::fence_barrier_init();
    // phase 0 never completes: no thread arrives
    tc::mbar_wait(&bar, 0, fault, tc::kFaultSelfTest, limit);
}

cudaError_t launch_selftest_wait(long long limit, int *fault, cudaStream_t s)
{
    k_selftest_wait<<<1, 32, 0, s>>>(limit, fault);
    return cudaGetLastError();
}

}  // namespace mhc
