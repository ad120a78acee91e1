// k3_shared.cu -- the always-on (shared) experts of the dense trunk, in bf16.
//
// Each MoE layer of the pages' model has two shared experts that run on
// every token ("Running Kimi K3 locally", "What are the four reductions, and
// why is the answer unchanged?"); like the rest of the dense trunk they stay
// in bf16 ("kimi-k3-in-c" explainer, "Why the trunk stays at 16 bits").  The
// form is the routed experts' SwiGLU, out[t] (+)= sum_s W_down^s
// (silu(W_gate^s x_t) * (W_up^s x_t)), with fp32 accumulation.
//
// At a few tokens per call the products are matrix-vector streams of bf16
// rows (2 bytes per weight, no decode: a bf16 is the high half of an fp32),
// so both kernels are bound by HBM: every lane loads 16 bytes (8 weights) of
// a row per step with several steps in flight, one warp per row, the tokens
// (gate/up) or h (down) held in shared memory.  Both are launched as
// programmatic dependents: their first weight rows are requested before the
// previous kernel on the stream has finished.
#include <cuda_runtime.h>

#include <algorithm>

#include "k3_device.cuh"
#include "k3_launch.cuh"

namespace k3 {

constexpr int SH_MAX = 4;     // shared experts per call at most
constexpr int SH_TMAX = 4;    // tokens per launch at most (x in shared memory)
constexpr int SH_WARPS = 16;  // warps per CTA
constexpr int SH_U = 4;       // 16-byte loads in flight per lane and matrix

struct SharedSrc {
    const uint16_t *gate[SH_MAX], *up[SH_MAX], *down[SH_MAX];
};

K3_DEV uint4 sh_ld16(const uint16_t *p) { return ld_stream16((const void *)p); }
// sum of the 8 bf16 weights of w times 8 fp32 values at v
K3_DEV float sh_dot8(uint4 w, const float *v, float acc)
{
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        acc = fmaf(__uint_as_float(q[i] << 16), v[2 * i], acc);
        acc = fmaf(__uint_as_float(q[i] & 0xffff0000u), v[2 * i + 1], acc);
    }
    return acc;
}

// h[t][s][r] = silu(gate_s[r] . x_t) * (up_s[r] . x_t), one warp per row
// q = s f + r; x [T][d] staged in shared memory.  d a multiple of 256.
__global__ void __launch_bounds__(SH_WARPS * 32) k3_shared_gateup(const SharedSrc src, int n, const float *x, int T,
                                                                  int d, int f, float *h)
{
    extern __shared__ float xs[];  // [T][d]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nc = d / 8;  // 16-byte chunks per row
    griddep_launch_dependents();
    const long nrows = (long)n * f, W = (long)gridDim.x * SH_WARPS;
    long q = (long)blockIdx.x * SH_WARPS + warp;
    // the first row's first chunks are requested before x can be read
    uint4 pg[SH_U], pu[SH_U];
    if (q < nrows) {
        const int s = (int)(q / f), r = (int)(q % f);
#pragma unroll
        for (int i = 0; i < SH_U; i++) {
            const int c = lane + 32 * i;
            pg[i] = c < nc ? sh_ld16(src.gate[s] + (size_t)r * d + 8 * c) : make_uint4(0, 0, 0, 0);
            pu[i] = c < nc ? sh_ld16(src.up[s] + (size_t)r * d + 8 * c) : make_uint4(0, 0, 0, 0);
        }
    }
    griddep_wait();  // x and h belong to the kernels around this one
    for (int i = threadIdx.x; i < T * d / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(xs)[i] = reinterpret_cast<const float4 *>(x)[i];
    __syncthreads();
    bool first = true;
    for (; q < nrows; q += W, first = false) {
        const int s = (int)(q / f), r = (int)(q % f);
        const uint16_t *gr = src.gate[s] + (size_t)r * d, *ur = src.up[s] + (size_t)r * d;
        float ag[SH_TMAX] = {}, au[SH_TMAX] = {};
        for (int c0 = 0; c0 < nc; c0 += 32 * SH_U) {
            uint4 wg[SH_U], wu[SH_U];
#pragma unroll
            for (int i = 0; i < SH_U; i++) {
                const int c = c0 + lane + 32 * i;
                if (first && c0 == 0) {
                    wg[i] = pg[i];
                    wu[i] = pu[i];
                } else {
                    wg[i] = c < nc ? sh_ld16(gr + 8 * c) : make_uint4(0, 0, 0, 0);
                    wu[i] = c < nc ? sh_ld16(ur + 8 * c) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int i = 0; i < SH_U; i++) {
                const int c = c0 + lane + 32 * i;
                if (c < nc) {
#pragma unroll
                    for (int t = 0; t < SH_TMAX; t++)
                        if (t < T) {
                            ag[t] = sh_dot8(wg[i], xs + (size_t)t * d + 8 * c, ag[t]);
                            au[t] = sh_dot8(wu[i], xs + (size_t)t * d + 8 * c, au[t]);
                        }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < SH_TMAX; t++)
            if (t < T) {
                const float g = warp_sum(ag[t]), u = warp_sum(au[t]);
                if (lane == 0) h[((size_t)t * n + s) * f + r] = silu(g) * u;
            }
    }
}

// out[t][c] (+)= sum_s down_s[c] . h[t][s], one warp per output row c; h
// [T][n][f] staged in shared memory.  f a multiple of 256.
__global__ void __launch_bounds__(SH_WARPS * 32) k3_shared_down(const SharedSrc src, int n, const float *h, int T,
                                                                int d, int f, float *out, int accumulate)
{
    extern __shared__ float hs[];  // [T][n][f]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nc = f / 8;
    griddep_launch_dependents();
    const long W = (long)gridDim.x * SH_WARPS;
    long c = (long)blockIdx.x * SH_WARPS + warp;
    uint4 pw[SH_U];
    if (c < d) {
#pragma unroll
        for (int i = 0; i < SH_U; i++) {
            const int k = lane + 32 * i;
            pw[i] = k < nc ? sh_ld16(src.down[0] + (size_t)c * f + 8 * k) : make_uint4(0, 0, 0, 0);
        }
    }
    griddep_wait();
    for (int i = threadIdx.x; i < T * n * f / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(hs)[i] = reinterpret_cast<const float4 *>(h)[i];
    __syncthreads();
    bool first = true;
    for (; c < d; c += W, first = false) {
        float acc[SH_TMAX] = {};
        for (int s = 0; s < n; s++) {
            const uint16_t *dr = src.down[s] + (size_t)c * f;
            for (int k0 = 0; k0 < nc; k0 += 32 * SH_U) {
                uint4 w[SH_U];
#pragma unroll
                for (int i = 0; i < SH_U; i++) {
                    const int k = k0 + lane + 32 * i;
                    if (first && s == 0 && k0 == 0)
                        w[i] = pw[i];
                    else
                        w[i] = k < nc ? sh_ld16(dr + 8 * k) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < SH_U; i++) {
                    const int k = k0 + lane + 32 * i;
                    if (k < nc) {
#pragma unroll
                        for (int t = 0; t < SH_TMAX; t++)
                            if (t < T) acc[t] = sh_dot8(w[i], hs + ((size_t)t * n + s) * f + 8 * k, acc[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < SH_TMAX; t++)
            if (t < T) {
                const float a = warp_sum(acc[t]);
                if (lane == 0) {
                    float *o = out + (size_t)t * d + c;
                    *o = accumulate ? *o + a : a;
                }
            }
    }
}

int num_sms();

bool shared_supported(int n, int d, int f)
{
    return n >= 1 && n <= SH_MAX && d % 256 == 0 && f % 256 == 0 && d <= 16384 && f <= 8192 &&
           (size_t)SH_TMAX * d * 4 <= 200 * 1024 && (size_t)SH_TMAX * n * f * 4 <= 200 * 1024;
}

// out (+)= the shared experts of T tokens, SH_TMAX tokens per launch pair;
// h: the workspace, SH_TMAX * n * f floats.
int launch_shared(const uint16_t *const *gate, const uint16_t *const *up, const uint16_t *const *down, int n,
                  const float *x, int T, int d, int f, float *h, float *out, int accumulate, cudaStream_t s)
{
    SharedSrc src = {};
    for (int i = 0; i < n; i++) {
        src.gate[i] = gate[i];
        src.up[i] = up[i];
        src.down[i] = down[i];
    }
    const int sms = num_sms();
    for (int t0 = 0; t0 < T; t0 += SH_TMAX) {
        const int tt = std::min(SH_TMAX, T - t0);
        const size_t sx = (size_t)tt * d * 4, sh = (size_t)tt * n * f * 4;
        if (ensure_smem((const void *)k3_shared_gateup, sx) != K3MOE_OK ||
            ensure_smem((const void *)k3_shared_down, sh) != K3MOE_OK)
            return K3MOE_ECUDA;
        const int g1 = (int)std::min<long>(((long)n * f + SH_WARPS - 1) / SH_WARPS, 4L * sms);
        const int g2 = (int)std::min<long>(((long)d + SH_WARPS - 1) / SH_WARPS, 4L * sms);
        if (launch_pdl(k3_shared_gateup, dim3(g1), dim3(SH_WARPS * 32), sx, s, src, n, x + (size_t)t0 * d, tt, d, f,
                       h) != cudaSuccess ||
            launch_pdl(k3_shared_down, dim3(g2), dim3(SH_WARPS * 32), sh, s, src, n, (const float *)h, tt, d, f,
                       out + (size_t)t0 * d, accumulate) != cudaSuccess) {
            cudaGetLastError();
            return K3MOE_ECUDA;
        }
    }
    return K3MOE_OK;
}
size_t shared_workspace_floats(int n, int f) { return (size_t)SH_TMAX * n * f; }

}  // namespace k3
