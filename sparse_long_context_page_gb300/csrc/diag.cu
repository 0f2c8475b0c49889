// Diagnostic: the bounded device wait that every kernel's mbarrier waits use,
// made to run out on purpose.  One block initialises an mbarrier that nothing
// arrives at, waits on it with the given limit (mbar_wait, as the kernels do)
// and, when the wait gives up, records MOIRA_DEV_TIMEOUT in the status word
// and returns.  No fault, trap or hang is involved: the kernel ends after
// `limit_ns` and the context stays usable.
#include "moira_device.cuh"
#include "moira_launch.h"

namespace moira {

__global__ void k_wait_timeout(uint32_t *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) unsigned long long s_bar;
    const uint32_t bar = smem_u32(&s_bar);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);                    // expects one arrival that never comes
        mbar_fence_init();
    }
    __syncthreads();
    if (!mbar_wait(bar, 0, limit_ns) && threadIdx.x == 0) raise_status(status, kDevTimeout);
}

cudaError_t launch_wait_timeout(uint32_t *status, unsigned long long limit_ns, cudaStream_t stream)
{
    k_wait_timeout<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace moira
