// Diagnostics of the device-side failure path: bounded waits made to run
// out on purpose.  No fault, trap or hang is involved: every wait gives up
// after its limit, records MOIRA_DEV_TIMEOUT in the status word and the
// kernel returns, so the context stays usable.
//  k_wait_timeout : one block waits on an mbarrier that nothing arrives at
//                   (the plain bounded wait);
//  k_wait_chain   : one block waits, through the kernels' WaitGuard, on
//                   `n_waits` such barriers in a row: the first wait runs out
//                   after the limit and every later one gives up at once;
//  k_barrier_timeout : `blocks` blocks meet at the kernels' inter-block
//                   barrier sized for one block more, which never completes.
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

constexpr int kChainBars = 64;

__global__ void k_wait_chain(uint32_t *status, unsigned long long limit_ns, int n_waits)
{
    __shared__ __align__(8) unsigned long long s_bar[kChainBars];
    __shared__ int s_abort;
    const WaitGuard wg{&s_abort, status};
    if (threadIdx.x == 0) {
        for (int i = 0; i < kChainBars; ++i) mbar_init(smem_u32(&s_bar[i]), 1);
        mbar_fence_init();
        s_abort = 0;                          // the chain itself must run out first
    }
    __syncthreads();
    for (int i = 0; i < n_waits; ++i) mbar_wait_g(smem_u32(&s_bar[i % kChainBars]), 0, wg, limit_ns);
}

__global__ void k_barrier_timeout(uint32_t *status, uint32_t *bar, unsigned long long limit_ns)
{
    __shared__ int s_abort;
    const WaitGuard wg{&s_abort, status};
    uint32_t gen = 0u;
    if (threadIdx.x == 0) {
        s_abort = 0;
        gen = barrier_generation(bar);
    }
    __syncthreads();
    group_barrier(bar, gridDim.x + 1u, gen, wg, limit_ns);
}

cudaError_t launch_wait_timeout(uint32_t *status, unsigned long long limit_ns, cudaStream_t stream)
{
    k_wait_timeout<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_wait_chain(uint32_t *status, unsigned long long limit_ns, int n_waits, cudaStream_t stream)
{
    k_wait_chain<<<1, 32, 0, stream>>>(status, limit_ns, n_waits);
    return cudaGetLastError();
}

cudaError_t launch_barrier_timeout(uint32_t *status, uint32_t *bar, int blocks, unsigned long long limit_ns,
                                   cudaStream_t stream)
{
    k_barrier_timeout<<<blocks, 32, 0, stream>>>(status, bar, limit_ns);
    return cudaGetLastError();
}

}  // namespace moira
