// k3_launch.cuh -- host-side launch helper shared by the kernels' launchers.
#pragma once
#include <cuda_runtime.h>

#include <atomic>

namespace k3 {

// Launches kernel<<<grid, block, smem, s>>>(args...) as a programmatic
// dependent of the previous kernel on s where the driver takes it (the
// kernel then overlaps its prologue, and the weight loads it issues before
// griddep_wait, with that kernel's tail), else as a plain launch.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args)
{
    static std::atomic<int> refused{0};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = refused.load(std::memory_order_relaxed) ? 0 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    if (e != cudaSuccess && cfg.numAttrs == 1) {
        cudaGetLastError();
        refused.store(1, std::memory_order_relaxed);
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kernel, args...);
    }
    return e;
}

}  // namespace k3
