// k3_selfcheck.cu -- runs the bounded-wait path of the kernels on purpose,
// without any fault: one CTA waits on an mbarrier that nothing will ever
// complete, gives up after the wait limit (2 s), records K3MOE_ETIMEOUT in the
// device error word and returns normally.  The GPU context stays usable.
#include <cuda_runtime.h>

#include "k3_device.cuh"

namespace k3 {
int *device_error_word();
}

namespace {
__global__ void k3_wait_on_nothing(int *err)
{
    __shared__ uint64_t bar;
    const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        k3::mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    k3::mbar_wait(b, 0, err);  // phase 0 never completes: returns false at the limit
}
}  // namespace

extern "C" int k3moe_check_wait_timeout(k3moe_stream s)
{
    int *err = k3::device_error_word();
    if (!err) return K3MOE_ECUDA;
    k3_wait_on_nothing<<<1, 32, 0, reinterpret_cast<cudaStream_t>(s)>>>(err);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}
