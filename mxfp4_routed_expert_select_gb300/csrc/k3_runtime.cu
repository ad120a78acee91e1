// k3_runtime.cu -- per-device host state shared by every launch of the
// library: the device error word, the SM count, and the dynamic shared-memory
// limits raised for each kernel.
//
// All three are kept per device (the current device at the call), since a
// CUDA context holds its own copy of each, and their first-time set-up is
// guarded so that concurrent first calls from several host threads are safe.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "k3_device.cuh"

// The device error word: one zero-initialised int in every device that loads
// the library, kept until the process exits.  No allocation is involved, so
// every entry point (the allocation-free one included) reports through it.
static __device__ int g_device_error;

namespace k3 {
namespace {
constexpr int kMaxDevices = 64;
std::once_flag g_err_once[kMaxDevices];
int *g_err_addr[kMaxDevices];
std::atomic<int> g_sms[kMaxDevices];
std::mutex g_smem_mu;
struct SmemLimit {
    int dev;
    const void *fn;
    size_t bytes;
};
std::vector<SmemLimit> g_smem;

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return -1;
    }
    return dev;
}
}  // namespace

// Device address of the error word on the current device (host code cannot
// use the symbol's name as an address); looked up once per device.
int *device_error_word()
{
    const int dev = current_device();
    if (dev < 0) return nullptr;
    std::call_once(g_err_once[dev], [dev] {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess)
            g_err_addr[dev] = (int *)p;
        else
            cudaGetLastError();
    });
    return g_err_addr[dev];
}

int num_sms()
{
    const int dev = current_device();
    if (dev < 0) return 1;
    int n = g_sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 1;
        }
        g_sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Raises kernel fn's dynamic shared-memory limit on the current device to at
// least `bytes` (once per device and size); K3MOE_ECUDA if refused.
int ensure_smem(const void *fn, size_t bytes)
{
    if (bytes <= 48 * 1024) return K3MOE_OK;
    const int dev = current_device();
    if (dev < 0) return K3MOE_ENODEV;
    std::lock_guard<std::mutex> lock(g_smem_mu);
    for (SmemLimit &l : g_smem)
        if (l.dev == dev && l.fn == fn) {
            if (l.bytes >= bytes) return K3MOE_OK;
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
                cudaGetLastError();
                return K3MOE_ECUDA;
            }
            l.bytes = bytes;
            return K3MOE_OK;
        }
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ECUDA;
    }
    g_smem.push_back({dev, fn, bytes});
    return K3MOE_OK;
}

}  // namespace k3
