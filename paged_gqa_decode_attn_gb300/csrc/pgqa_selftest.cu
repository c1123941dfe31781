// Self-test of the kernels' bounded waits.  One CTA waits on an mbarrier that
// nothing arrives on, through the same mbar_wait_bounded the split, prefill
// and prep kernels use.  After about one second of SM clock the wait gives
// up, ORs kErrTimeoutFull into the library's device error word and returns,
// so the failure path of every bounded wait is exercised with no fault, no
// trap and no hang, and the context stays usable.
#include "pgqa_device.cuh"

namespace pgqa {

namespace {

__global__ void __launch_bounds__(32) bounded_wait_probe_kernel(unsigned int *err)
{
    __shared__ unsigned long long bar;
    if (threadIdx.x != 0)
        return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    mbar_init_fence();
    mbar_wait_bounded(b, 0, err, kErrTimeoutFull);   // phase 0 never completes: gives up
}

}  // namespace

cudaError_t launch_bounded_wait_probe(unsigned int *err, cudaStream_t stream)
{
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace pgqa
