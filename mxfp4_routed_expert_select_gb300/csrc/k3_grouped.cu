// k3_grouped.cu -- grouped MXFP4 products for multi-token batches (sm_103a).
//
// After routing, the T*k (token, slot) pairs are grouped by expert (k3_group).
// Each work item is (expert, up to NT pairs of that expert); a unit is an
// item times a block of RB rows.  A persistent grid walks the units.
//
// Per unit the CTA holds the NT activation rows in registers: lane l of warp
// w owns the 16 input columns of half-group (32 w + l), so a row of weights
// is read once (8 bytes per lane, coalesced 256 B per warp) and multiplied
// into all NT activations while it is in registers.  Partials are reduced
// across lanes (transpose reduction) and across warps (shared memory).
//
//   MODE_GATEUP: h[p][r] = silu(gate_e[r] . x_t) * (up_e[r] . x_t)
//   MODE_DOWN  : Y[p][i] = w_p * (down_e[i] . h[p])
// and k3_combine sums Y over a token's k slots in slot order.
#include "k3_device.cuh"

namespace k3 {

int num_sms();

constexpr int MODE_GATEUP = 1, MODE_DOWN = 0;

template <typename XT>
K3_DEV void load16(const XT *p, float2 (&v)[8]);
template <>
K3_DEV void load16<float>(const float *p, float2 (&v)[8])
{
    const float4 *q = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float4 a = __ldg(q + i);
        v[2 * i] = make_float2(a.x, a.y);
        v[2 * i + 1] = make_float2(a.z, a.w);
    }
}
template <>
K3_DEV void load16<__nv_bfloat16>(const __nv_bfloat16 *p, float2 (&v)[8])
{
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 2; i++) {
        uint4 a = __ldg(q + i);
        uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; j++)
            v[4 * i + j] = make_float2(__uint_as_float(w[j] << 16),
                                       __uint_as_float(w[j] & 0xffff0000u));
    }
}

template <int NT, int U, int MODE, typename XT>
__global__ void __launch_bounds__(512) k3_grouped_rows(
    const XT *__restrict__ xin,          // GATEUP: X [T][d]; DOWN: h [pairs][f] (fp32)
    const DevExpert *__restrict__ table, const int32_t *__restrict__ perm,
    const int4 *__restrict__ items, const int32_t *__restrict__ n_items_p, int k, int in,
    int rows, int RB, const float *__restrict__ wsel, float *__restrict__ out)
{
    extern __shared__ float red[];  // [nwarps][RB][NT][2]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int HG = in >> 4;
    const int hg = warp * 32 + lane;
    const bool active = hg < HG;
    const int nrb = (rows + RB - 1) / RB;
    const int n_units = (*n_items_p) * nrb;
    const size_t rowB = (size_t)(in >> 1), rowS = (size_t)(in >> 5);
    constexpr int NM = (MODE == MODE_GATEUP) ? 2 : 1;
    constexpr int NV = NM * NT * U;
    static_assert((NV & (NV - 1)) == 0 && NV <= 32, "NV must be a power of two <= 32");

    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
        const int it = unit / nrb, rb = unit - it * nrb;
        const int4 item = items[it];
        const int e = item.x, off = item.y, n = item.z;
        const int r0 = rb * RB, r1 = min(r0 + RB, rows);
        const DevExpert ex = table[e];
        const uint8_t *P0 = (MODE == MODE_GATEUP) ? ex.gp : ex.dp;
        const uint8_t *S0 = (MODE == MODE_GATEUP) ? ex.gs : ex.ds;
        const uint8_t *P1 = ex.up;
        const uint8_t *S1 = ex.us;

        int pr[NT];
        float2 xr[NT][8];
#pragma unroll
        for (int i = 0; i < NT; i++) {
            pr[i] = (i < n) ? perm[off + i] : -1;
#pragma unroll
            for (int q = 0; q < 8; q++) xr[i][q] = make_float2(0.f, 0.f);
            if (active && i < n) {
                const size_t src_row = (MODE == MODE_GATEUP) ? (size_t)(pr[i] / k) : (size_t)pr[i];
                load16<XT>(xin + src_row * in + 16 * hg, xr[i]);
            }
        }

        for (int c = r0; c < r1; c += U) {
            uint2 qa[U], qb[U];
            uint32_t sa[U], sb[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int r = c + u;
                qa[u] = make_uint2(0, 0);
                qb[u] = make_uint2(0, 0);
                sa[u] = 255;
                sb[u] = 255;
                if (active && r < r1) {
                    qa[u] = ld_stream8(P0 + r * rowB + 8 * (size_t)hg);
                    sa[u] = ld_stream_u8(S0 + r * rowS + (hg >> 1));
                    if (MODE == MODE_GATEUP) {
                        qb[u] = ld_stream8(P1 + r * rowB + 8 * (size_t)hg);
                        sb[u] = ld_stream_u8(S1 + r * rowS + (hg >> 1));
                    }
                }
            }
            float v[NV];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const float sca = e8m0_scale(sa[u]);
                const float scb = e8m0_scale(sb[u]);
#pragma unroll
                for (int i = 0; i < NT; i++) {
                    v[(0 * NT + i) * U + u] = (sa[u] == 255u) ? 0.f : dot16(qa[u], xr[i]) * sca;
                    if (MODE == MODE_GATEUP)
                        v[(1 * NT + i) * U + u] =
                            (sb[u] == 255u) ? 0.f : dot16(qb[u], xr[i]) * scb;
                }
            }
            warp_transpose_reduce<NV>(v, lane);
            constexpr int LPV = 32 / NV;
            if ((lane % LPV) == 0) {
                const int vi = sel_of<NV>(lane);
                const int u = vi % U;
                const int i = (vi / U) % NT;
                const int m = vi / (U * NT);
                const int r = c + u;
                if (r < r1) red[(((size_t)warp * RB + (r - r0)) * NT + i) * 2 + m] = v[0];
            }
        }
        __syncthreads();
        const int nrow = r1 - r0;
        for (int idx = threadIdx.x; idx < nrow * NT; idx += blockDim.x) {
            const int rr = idx / NT, i = idx % NT;
            if (i >= n) continue;
            float a = 0.f, b = 0.f;
            for (int w = 0; w < nwarps; w++) {
                a += red[(((size_t)w * RB + rr) * NT + i) * 2 + 0];
                if (MODE == MODE_GATEUP) b += red[(((size_t)w * RB + rr) * NT + i) * 2 + 1];
            }
            const int p = perm[off + i];
            if (MODE == MODE_GATEUP)
                out[(size_t)p * rows + r0 + rr] = silu(a) * b;
            else
                out[(size_t)p * rows + r0 + rr] = a * wsel[p];
        }
        __syncthreads();
    }
}

// out[t][i] = sum_j Y[t*k + j][i], slots in order.
__global__ void k3_combine(const float *__restrict__ Y, int T, int k, int d, float *__restrict__ out)
{
    const size_t n4 = (size_t)T * d / 4;
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n4;
         q += (size_t)gridDim.x * blockDim.x) {
        const size_t t = (4 * q) / d, i = (4 * q) % d;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; j++) {
            float4 y = *reinterpret_cast<const float4 *>(Y + ((t * k + j) * d + i));
            a.x += y.x; a.y += y.y; a.z += y.z; a.w += y.w;
        }
        *reinterpret_cast<float4 *>(out + t * d + i) = a;
    }
}

// ------------------------------------------------------------- launchers

constexpr int GNT = 4;  // pairs per item

template <int NT, int U, int MODE, typename XT>
static int launch_one(const XT *xin, const DevExpert *table, const int32_t *perm,
                      const int4 *items, const int32_t *n_items, int max_items, int k, int in,
                      int rows, int RB, const float *wsel, float *out, cudaStream_t s)
{
    const int HG = in / 16;
    const int nwarps = (HG + 31) / 32;
    if (nwarps > 16) return K3MOE_EINVAL;
    const int threads = nwarps * 32;
    const size_t smem = (size_t)nwarps * RB * NT * 2 * sizeof(float);
    auto kern = k3_grouped_rows<NT, U, MODE, XT>;
    if (ensure_smem((const void *)kern, smem) != K3MOE_OK) return K3MOE_ECUDA;
    int bps = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, threads, smem);
    if (bps < 1) bps = 1;
    const long units_max = (long)max_items * ((rows + RB - 1) / RB);
    long grid = (long)num_sms() * bps;
    if (grid > units_max) grid = units_max;
    if (grid < 1) grid = 1;
    kern<<<(int)grid, threads, smem, s>>>(xin, table, perm, items, n_items, k, in, rows, RB, wsel,
                                          out);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int grouped_nt() { return GNT; }

int launch_grouped_gateup(const void *X, int xdt, const DevExpert *table, const int32_t *perm,
                          const int4 *items, const int32_t *n_items, int max_items, int k, int d,
                          int f, float *h, cudaStream_t s)
{
    const int RB = 32;
    if (xdt == K3MOE_F32)
        return launch_one<GNT, 2, MODE_GATEUP, float>((const float *)X, table, perm, items,
                                                      n_items, max_items, k, d, f, RB, nullptr,
                                                      h, s);
    return launch_one<GNT, 2, MODE_GATEUP, __nv_bfloat16>((const __nv_bfloat16 *)X, table, perm,
                                                          items, n_items, max_items, k, d, f, RB,
                                                          nullptr, h, s);
}

int launch_grouped_down(const float *h, const DevExpert *table, const int32_t *perm,
                        const int4 *items, const int32_t *n_items, int max_items, int k, int d,
                        int f, const float *wsel, float *Y, cudaStream_t s)
{
    const int RB = 64;
    return launch_one<GNT, 4, MODE_DOWN, float>(h, table, perm, items, n_items, max_items, k, f,
                                                d, RB, wsel, Y, s);
}

int launch_combine(const float *Y, int T, int k, int d, float *out, cudaStream_t s)
{
    const size_t n4 = (size_t)T * d / 4;
    int grid = (int)((n4 + 255) / 256);
    if (grid > 4 * num_sms()) grid = 4 * num_sms();
    if (grid < 1) grid = 1;
    k3_combine<<<grid, 256, 0, s>>>(Y, T, k, d, out);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

// --------------------------------------------------------- norm / residual

__global__ void k3_rmsnorm_kernel(float *u, const float *x, int n, float eps)
{
    __shared__ float part[32];
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(x[i], x[i], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = (threadIdx.x < (blockDim.x >> 5)) ? part[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) part[0] = v;
    }
    __syncthreads();
    const float inv = rsqrtf(part[0] / (float)n + eps);
    for (int i = threadIdx.x; i < n; i += blockDim.x) u[i] = x[i] * inv;
}

__global__ void k3_residual_kernel(float *x, const float *dlt, int n)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        x[i] += dlt[i];
}

int launch_rmsnorm(float *u, const float *x, int n, float eps, cudaStream_t s)
{
    k3_rmsnorm_kernel<<<1, 1024, 0, s>>>(u, x, n, eps);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int launch_residual(float *x, const float *dlt, int n, cudaStream_t s)
{
    int grid = (n + 255) / 256;
    if (grid > 1024) grid = 1024;
    k3_residual_kernel<<<grid, 256, 0, s>>>(x, dlt, n);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

}  // namespace k3
