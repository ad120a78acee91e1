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
// so both kernels are bound by HBM and by how many of their loads are in
// flight: every lane requests all of its 16-byte chunks of a unit at once
// (gate/up: four rows split along K over the CTA's warps; down: one output
// row per warp), the next unit's before the current one is reduced, the
// tokens (gate/up) or h (down) held in shared memory, and the grids are one
// resident wave.  Both are launched as programmatic dependents: their first
// weight rows are requested before the previous kernel on the stream has
// finished.
#include <cuda_runtime.h>

#include <algorithm>

#include "k3_device.cuh"
#include "k3_launch.cuh"

namespace k3 {

constexpr int SH_MAX = 4;     // shared experts per call at most
constexpr int SH_TMAX = 4;    // tokens per launch at most (x in shared memory)
constexpr int SH_WARPS = 16;  // warps per CTA
constexpr int SH_RG = 4;      // gate/up rows per unit
constexpr int SH_CH = 2;      // 16-byte chunks per lane and row of a gate/up K-slice (d <= 8192)
constexpr int SH_CHD = 16;    // 16-byte chunks per lane of a down row (n f <= 4096)

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

// h[t][s][r] = silu(gate_s[r] . x_t) * (up_s[r] . x_t).  A unit is SH_RG rows
// q = s f + r (of one expert: f % SH_RG == 0); warp w of the CTA takes K-slice
// w of them (d / 8 / SH_WARPS chunks of 8 weights), every lane issuing all of
// its loads for the unit at once, so that a row costs one memory round trip
// instead of one per chunk; the slices' partial sums meet in shared memory.
// x [T][d] is staged in shared memory.
__global__ void __launch_bounds__(SH_WARPS * 32) k3_shared_gateup(const SharedSrc src, int n, const float *x, int T,
                                                                  int d, int f, float *h)
{
    extern __shared__ float xs[];  // [T][d], then red [SH_WARPS][SH_RG * 2 * SH_TMAX]
    float *red = xs + (size_t)T * d;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cpw = d / 8 / SH_WARPS;  // chunks per warp slice
    const int nunits = n * f / SH_RG;
    griddep_launch_dependents();
    int u = blockIdx.x;
    // the first unit's weights are requested before x can be read
    uint4 wg[SH_RG][SH_CH], wu[SH_RG][SH_CH];
    auto load = [&](int uu) {
        const int q0 = uu * SH_RG, s = q0 / f, r0 = q0 % f;
#pragma unroll
        for (int r = 0; r < SH_RG; r++)
#pragma unroll
            for (int c = 0; c < SH_CH; c++) {
                const int ch = lane + 32 * c;
                const size_t off = (size_t)(r0 + r) * d + 8 * (size_t)(warp * cpw + ch);
                wg[r][c] = ch < cpw ? sh_ld16(src.gate[s] + off) : make_uint4(0, 0, 0, 0);
                wu[r][c] = ch < cpw ? sh_ld16(src.up[s] + off) : make_uint4(0, 0, 0, 0);
            }
    };
    if (u < nunits) load(u);
    griddep_wait();  // x and h belong to the kernels around this one
    for (int i = threadIdx.x; i < T * d / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(xs)[i] = reinterpret_cast<const float4 *>(x)[i];
    __syncthreads();
    constexpr int NV = SH_RG * 2 * SH_TMAX;  // (row, matrix, token) partial sums of a lane
    for (; u < nunits; u += gridDim.x) {
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; i++) v[i] = 0.f;
#pragma unroll
        for (int c = 0; c < SH_CH; c++) {
            const int ch = lane + 32 * c;
            if (ch < cpw) {
                const int col = 8 * (warp * cpw + ch);
#pragma unroll
                for (int t = 0; t < SH_TMAX; t++)
                    if (t < T) {
#pragma unroll
                        for (int r = 0; r < SH_RG; r++) {
                            v[(r * 2 + 0) * SH_TMAX + t] = sh_dot8(wg[r][c], xs + (size_t)t * d + col, v[(r * 2 + 0) * SH_TMAX + t]);
                            v[(r * 2 + 1) * SH_TMAX + t] = sh_dot8(wu[r][c], xs + (size_t)t * d + col, v[(r * 2 + 1) * SH_TMAX + t]);
                        }
                    }
            }
        }
        // the next unit's weights are requested before this one is reduced
        const int un = u + gridDim.x;
        if (un < nunits) load(un);
        warp_transpose_reduce<NV>(v, lane);  // lane l: the warp's sum of value sel_of(l) = l
        red[warp * NV + lane] = v[0];
        __syncthreads();
        if ((int)threadIdx.x < SH_RG * T) {
            const int r = threadIdx.x / T, t = threadIdx.x % T;
            float g = 0.f, up = 0.f;
            for (int w2 = 0; w2 < SH_WARPS; w2++) {
                g += red[w2 * NV + (r * 2 + 0) * SH_TMAX + t];
                up += red[w2 * NV + (r * 2 + 1) * SH_TMAX + t];
            }
            const int q = u * SH_RG + r, s = q / f;
            h[((size_t)t * n + s) * f + (q % f)] = silu(g) * up;
        }
        __syncthreads();
    }
}

// out[t][c] (+)= sum_s down_s[c] . h[t][s], one warp per output row c at a
// time with every 16-byte chunk of the row (n f bf16 weights) requested at
// once; h [T][n][f] staged in shared memory.
__global__ void __launch_bounds__(SH_WARPS * 32) k3_shared_down(const SharedSrc src, int n, const float *h, int T,
                                                                int d, int f, float *out, int accumulate)
{
    extern __shared__ float hs[];  // [T][n][f]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ncs = f / 8;          // chunks per row of one expert
    const int nch = n * ncs;        // chunks of an output row
    griddep_launch_dependents();
    const int W = gridDim.x * SH_WARPS;
    int c = blockIdx.x * SH_WARPS + warp;
    uint4 w[SH_CHD];
    auto load = [&](int row) {
#pragma unroll
        for (int i = 0; i < SH_CHD; i++) {
            const int ch = lane + 32 * i;
            w[i] = ch < nch ? sh_ld16(src.down[ch / ncs] + (size_t)row * f + 8 * (ch % ncs)) : make_uint4(0, 0, 0, 0);
        }
    };
    if (c < d) load(c);
    griddep_wait();
    for (int i = threadIdx.x; i < T * n * f / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(hs)[i] = reinterpret_cast<const float4 *>(h)[i];
    __syncthreads();
    for (; c < d; c += W) {
        float acc[SH_TMAX];
#pragma unroll
        for (int t = 0; t < SH_TMAX; t++) acc[t] = 0.f;
#pragma unroll
        for (int i = 0; i < SH_CHD; i++) {
            const int ch = lane + 32 * i;
            if (ch < nch) {
                const int s = ch / ncs, k = ch % ncs;
#pragma unroll
                for (int t = 0; t < SH_TMAX; t++)
                    if (t < T) acc[t] = sh_dot8(w[i], hs + ((size_t)t * n + s) * f + 8 * k, acc[t]);
            }
        }
        if (c + W < d) load(c + W);
        warp_transpose_reduce<SH_TMAX>(acc, lane);
        constexpr int LPV = 32 / SH_TMAX;
        if ((lane % LPV) == 0) {
            const int t = sel_of<SH_TMAX>(lane);
            if (t < T) {
                float *o = out + (size_t)t * d + c;
                *o = accumulate ? *o + acc[0] : acc[0];
            }
        }
    }
}

// The same product with two rows in flight per warp (n f <= 3072): the
// loads of row c + 2W are issued as soon as row c is multiplied, so every
// warp keeps the next row's loads outstanding while it works on one; eight
// warps a CTA and two CTAs an SM hold as many rows in registers as the
// register file allows.
constexpr int SH2_WARPS = 8;
constexpr int SH2_CH = 12;  // 16-byte chunks per lane of a down row (n f <= 3072)

__global__ void __launch_bounds__(SH2_WARPS * 32, 2) k3_shared_down2(const SharedSrc src, int n, const float *h, int T,
                                                                    int d, int f, float *out, int accumulate)
{
    extern __shared__ float hs[];  // [T][n][f]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ncs = f / 8;    // chunks per row of one expert
    const int nch = n * ncs;  // chunks of an output row
    griddep_launch_dependents();
    const int W = gridDim.x * SH2_WARPS;
    int c = blockIdx.x * SH2_WARPS + warp;
    uint4 w0[SH2_CH], w1[SH2_CH];
    auto load = [&](uint4(&w)[SH2_CH], int row) {
#pragma unroll
        for (int i = 0; i < SH2_CH; i++) {
            const int ch = lane + 32 * i;
            w[i] = ch < nch ? sh_ld16(src.down[ch / ncs] + (size_t)row * f + 8 * (ch % ncs)) : make_uint4(0, 0, 0, 0);
        }
    };
    auto dots = [&](const uint4(&w)[SH2_CH], float(&acc)[SH_TMAX]) {
#pragma unroll
        for (int t = 0; t < SH_TMAX; t++) acc[t] = 0.f;
#pragma unroll
        for (int i = 0; i < SH2_CH; i++) {
            const int ch = lane + 32 * i;
            if (ch < nch) {
                const int s = ch / ncs, k = ch % ncs;
#pragma unroll
                for (int t = 0; t < SH_TMAX; t++)
                    if (t < T) acc[t] = sh_dot8(w[i], hs + ((size_t)t * n + s) * f + 8 * k, acc[t]);
            }
        }
    };
    auto finish = [&](float(&acc)[SH_TMAX], int row) {
        warp_transpose_reduce<SH_TMAX>(acc, lane);
        constexpr int LPV = 32 / SH_TMAX;
        if ((lane % LPV) == 0) {
            const int t = sel_of<SH_TMAX>(lane);
            if (t < T) {
                float *o = out + (size_t)t * d + row;
                *o = accumulate ? *o + acc[0] : acc[0];
            }
        }
    };
    if (c < d) load(w0, c);
    if (c + W < d) load(w1, c + W);
    griddep_wait();
    for (int i = threadIdx.x; i < T * n * f / 4; i += blockDim.x)
        reinterpret_cast<float4 *>(hs)[i] = reinterpret_cast<const float4 *>(h)[i];
    __syncthreads();
    for (; c < d; c += 2 * W) {
        float acc[SH_TMAX];
        dots(w0, acc);  // row c
        if (c + 2 * W < d) load(w0, c + 2 * W);
        finish(acc, c);
        if (c + W >= d) break;
        dots(w1, acc);  // row c + W
        if (c + 3 * W < d) load(w1, c + 3 * W);
        finish(acc, c + W);
    }
}

int num_sms();

bool shared_supported(int n, int d, int f)
{
    return n >= 1 && n <= SH_MAX && d % 256 == 0 && f % 256 == 0 && d <= 8192 && (size_t)n * f <= 32 * SH_CHD * 8 &&
           (d / 8) % SH_WARPS == 0 && (size_t)SH_TMAX * d * 4 + SH_WARPS * SH_RG * 2 * SH_TMAX * 4 <= 200 * 1024 &&
           (size_t)SH_TMAX * n * f * 4 <= 200 * 1024;
}

template <typename K>
static int resident_grid(K kernel, size_t smem, long want, int threads = SH_WARPS * 32)
{
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem) != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    return (int)std::max(1L, std::min<long>(want, (long)b * num_sms()));
}

// out (+)= the shared experts of T tokens, SH_TMAX tokens per launch pair;
// h: the workspace, SH_TMAX * n * f floats.  Both grids are as large as can
// be resident at once (one wave).
int launch_shared(const uint16_t *const *gate, const uint16_t *const *up, const uint16_t *const *down, int n,
                  const float *x, int T, int d, int f, float *h, float *out, int accumulate, cudaStream_t s)
{
    SharedSrc src = {};
    for (int i = 0; i < n; i++) {
        src.gate[i] = gate[i];
        src.up[i] = up[i];
        src.down[i] = down[i];
    }
    for (int t0 = 0; t0 < T; t0 += SH_TMAX) {
        const int tt = std::min(SH_TMAX, T - t0);
        const size_t sx = (size_t)tt * d * 4 + SH_WARPS * SH_RG * 2 * SH_TMAX * 4, sh = (size_t)tt * n * f * 4;
        const bool two = (long)n * f <= 32L * SH2_CH * 8;  // two rows in flight per warp
        if (ensure_smem((const void *)k3_shared_gateup, sx) != K3MOE_OK ||
            ensure_smem(two ? (const void *)k3_shared_down2 : (const void *)k3_shared_down, sh) != K3MOE_OK)
            return K3MOE_ECUDA;
        const int g1 = resident_grid(k3_shared_gateup, sx, (long)n * f / SH_RG);
        cudaError_t e = launch_pdl(k3_shared_gateup, dim3(g1), dim3(SH_WARPS * 32), sx, s, src, n,
                                   x + (size_t)t0 * d, tt, d, f, h);
        if (e == cudaSuccess) {
            if (two) {
                const int g2 = resident_grid(k3_shared_down2, sh, ((long)d + SH2_WARPS - 1) / SH2_WARPS, SH2_WARPS * 32);
                e = launch_pdl(k3_shared_down2, dim3(g2), dim3(SH2_WARPS * 32), sh, s, src, n, (const float *)h, tt, d,
                               f, out + (size_t)t0 * d, accumulate);
            } else {
                const int g2 = resident_grid(k3_shared_down, sh, ((long)d + SH_WARPS - 1) / SH_WARPS);
                e = launch_pdl(k3_shared_down, dim3(g2), dim3(SH_WARPS * 32), sh, s, src, n, (const float *)h, tt, d,
                               f, out + (size_t)t0 * d, accumulate);
            }
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            return K3MOE_ECUDA;
        }
    }
    return K3MOE_OK;
}
size_t shared_workspace_floats(int n, int f) { return (size_t)SH_TMAX * n * f; }

}  // namespace k3
