// k3_noalloc.cu -- k3moe_expert_gemv_noalloc: the single-expert product for
// callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or anything that does) on the call
// path: code that runs while a stream is being captured in global capture
// mode, latency-critical threads with a no-allocation rule, plug-ins that must
// not touch the host application's allocator, or systems whose device memory
// is budgeted once at start-up.  This entry point gives them the same result
// as k3moe_expert_gemv without a workspace argument: the SwiGLU intermediate h
// lives in a fixed file-scope device array.  Errors found on the device (a
// bounded wait that ran out) go to the library's device error word, which is
// itself a file-scope device variable, and k3moe_device_error() reads them.
//
// The array exists once per device that loads the library and stays allocated
// until the process exits.  Host code cannot use its name as a device address
// (in host code the name denotes a host-side stand-in), so the first call on
// each device, with that device current, looks the address up with
// cudaGetSymbolAddress and remembers it; make that first call before any
// stream capture.  Every call on a device shares the same array: two calls
// whose kernels overlap on the GPU race on h, so serialise them (one stream,
// or events).  h is overwritten completely by every call before it is read,
// so nothing has to be cleared between calls.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "k3_device.cuh"

namespace k3 {
int launch_rows_t1_err(int mode, const float *x, const ExpertSrc &src, int k, int in, int rows,
                       float *out, int *err, cudaStream_t s);
int launch_down_t1(const float *h, const ExpertSrc &src, const float *w, int k, int d, int f,
                   float *out, cudaStream_t s, bool acc = false);
}  // namespace k3

// Largest expert intermediate size f the static scratch holds (8 KB of fp32).
#define K3_NOALLOC_MAX_F K3MOE_NOALLOC_MAX_F

static __device__ __align__(256) float g_noalloc_h[K3_NOALLOC_MAX_F];

namespace {
constexpr int kMaxDevices = 64;
std::once_flag g_h_once[kMaxDevices];
float *g_h_addr[kMaxDevices];

// Device addresses of h and of the device error word on the current device
// (looked up once per device; concurrent first calls are safe).
int noalloc_setup(float **h, int **err)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return K3MOE_ENODEV;
    }
    std::call_once(g_h_once[dev], [dev] {
        void *ph = nullptr;
        if (cudaGetSymbolAddress(&ph, g_noalloc_h) == cudaSuccess)
            g_h_addr[dev] = (float *)ph;
        else
            cudaGetLastError();
    });
    *h = g_h_addr[dev];
    *err = k3::device_error_word();
    return *h && *err ? K3MOE_OK : K3MOE_ECUDA;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool valid_mat(const k3moe_mat &m, int rows, int in)
{
    return m.packed && m.scales && aligned16(m.packed) && aligned16(m.scales) && m.rows == rows &&
           m.in == in;
}
}  // namespace

extern "C" int k3moe_expert_gemv_noalloc(float *y, const float *x, const k3moe_expert *e,
                                         int32_t d, int32_t f, k3moe_stream s)
{
    if (!y || !x || !e) return K3MOE_EINVAL;
    if (d <= 0 || f <= 0 || d % 32 || f % 32 || d > 16384 || f > K3_NOALLOC_MAX_F)
        return K3MOE_EINVAL;
    if (!valid_mat(e->gate, f, d) || !valid_mat(e->up, f, d) || !valid_mat(e->down, d, f) ||
        !aligned16(y) || !aligned16(x))
        return K3MOE_EINVAL;
    float *h = nullptr;
    int *err = nullptr;
    const int st = noalloc_setup(&h, &err);
    if (st != K3MOE_OK) return st;
    k3::ExpertSrc src;
    memset(&src, 0, sizeof(src));
    src.inl[0] = {e->gate.packed, e->gate.scales, e->up.packed, e->up.scales, e->down.packed,
                  e->down.scales};
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    const int r = k3::launch_rows_t1_err(1, x, src, 1, d, f, h, err, cs);
    if (r != K3MOE_OK) return r;
    return k3::launch_down_t1(h, src, nullptr, 1, d, f, y, cs);
}
