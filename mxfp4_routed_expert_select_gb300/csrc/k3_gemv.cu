// k3_gemv.cu -- batch-1 MXFP4 expert kernels (sm_103a).
//
//   k3_rows_t1   : gate/up products + SwiGLU for k selected experts (or one
//                  plain matrix, the pages' k3_matmul_mxfp4 primitive)
//   k3_down_t1   : down products of k experts with the weighted combine
//
// Memory-bound design (about 1.9 weights per byte of HBM traffic):
//   - one lane owns one 32-group of columns for the whole kernel and keeps
//     those 32 activations in registers, so the activation vector is read
//     once per CTA and never again;
//   - a warp reads 512 contiguous bytes of a row per load (16 B per lane,
//     exactly one group), streamed with L1 no-allocate hints; the 32 E8M0
//     bytes of the same groups come in one 32-byte sector;
//   - U rows are loaded before any is used, to keep enough bytes in flight;
//   - per-lane partials of U rows are reduced across the warp with a
//     transpose reduction (one shuffle per row instead of five), then across
//     warps in shared memory;
//   - the grid is sized to the SM count times the resident CTAs per SM, with
//     an equal row range per CTA, so every SM streams the same bytes.
#include "k3_device.cuh"

namespace k3 {

// ---------------------------------------------------------------- gate / up
// MODE 0: y[q] = W x for one matrix (W given in src.inl[0].gp/.gs, k = 1).
// MODE 1: h[j][r] = silu(gate_j[r] . x) * (up_j[r] . x), q = j * f + r.
template <int MODE, int U>
__global__ void __launch_bounds__(512) k3_rows_t1(const float *__restrict__ x, ExpertSrc src,
                                                   int k, int in, int rows, float *__restrict__ out,
                                                   int rows_per_cta)
{
    extern __shared__ float red[];  // [nwarps][rows_per_cta][2]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int G = in >> 5;
    const int g = warp * 32 + lane;
    const bool active = g < G;

    float2 xr[16];
#pragma unroll
    for (int i = 0; i < 16; i++) xr[i] = make_float2(0.f, 0.f);
    if (active) {
        const float4 *xp = reinterpret_cast<const float4 *>(x + 32 * g);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            float4 v = __ldg(xp + i);
            xr[2 * i] = make_float2(v.x, v.y);
            xr[2 * i + 1] = make_float2(v.z, v.w);
        }
    }

    const long total = (long)k * rows;
    const long q0 = (long)blockIdx.x * rows_per_cta;
    const long q1 = min(q0 + rows_per_cta, total);
    const size_t rowB = (size_t)(in >> 1), rowS = (size_t)G;
    constexpr int NV = (MODE == 1) ? 2 * U : U;

    for (long c = q0; c < q1; c += U) {
        uint4 qa[U], qb[U];
        uint32_t sa[U], sb[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const long q = c + u;
            qa[u] = make_uint4(0, 0, 0, 0);
            qb[u] = make_uint4(0, 0, 0, 0);
            sa[u] = 255;
            sb[u] = 255;
            if (active && q < q1) {
                const int j = (int)(q / rows);
                const int r = (int)(q - (long)j * rows);
                const DevExpert e = fetch_expert(src, j);
                qa[u] = ld_stream16(e.gp + r * rowB + 16 * (size_t)g);
                sa[u] = ld_stream_u8(e.gs + r * rowS + g);
                if (MODE == 1) {
                    qb[u] = ld_stream16(e.up + r * rowB + 16 * (size_t)g);
                    sb[u] = ld_stream_u8(e.us + r * rowS + g);
                }
            }
        }
        float v[NV];
#pragma unroll
        for (int u = 0; u < U; u++) {
            v[u] = (sa[u] == 255u) ? 0.f : dot32(qa[u], xr) * e8m0_scale(sa[u]);
            if (MODE == 1) v[U + u] = (sb[u] == 255u) ? 0.f : dot32(qb[u], xr) * e8m0_scale(sb[u]);
        }
        warp_transpose_reduce<NV>(v, lane);
        constexpr int LPV = 32 / NV;  // lanes holding each value
        if ((lane % LPV) == 0) {
            const int vi = sel_of<NV>(lane);
            const int u = (MODE == 1) ? (vi % U) : vi;
            const int which = (MODE == 1) ? (vi / U) : 0;
            const long q = c + u;
            if (q < q1) red[((size_t)warp * rows_per_cta + (q - q0)) * 2 + which] = v[0];
        }
    }
    __syncthreads();
    for (long t = threadIdx.x; t < q1 - q0; t += blockDim.x) {
        float a = 0.f, b = 0.f;
        for (int w = 0; w < nwarps; w++) {
            a += red[((size_t)w * rows_per_cta + t) * 2 + 0];
            if (MODE == 1) b += red[((size_t)w * rows_per_cta + t) * 2 + 1];
        }
        out[q0 + t] = (MODE == 1) ? silu(a) * b : a;
    }
}

// -------------------------------------------------------------------- down
// out[i] = sum_j w[j] * (down_j[i] . h[j])  over the k selected experts.
// CTA: k * nsub warps; warp (j, s) handles expert j and rows i0+s, i0+s+nsub..
// Lane owns HPL half-groups (16 columns each) of the f-long input.
template <int HPL, int U>
__global__ void __launch_bounds__(512) k3_down_t1(const float *__restrict__ h, ExpertSrc src,
                                                  const float *__restrict__ w, int k, int d, int f,
                                                  float *__restrict__ out, int rows_per_cta)
{
    extern __shared__ float red[];  // [k][rows_per_cta]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsub = (blockDim.x >> 5) / k;
    const int j = warp % k, s = warp / k;
    const int HG = f >> 4;
    const int i0 = blockIdx.x * rows_per_cta;
    const int i1 = min(i0 + rows_per_cta, d);

    if (s < nsub) {
        const DevExpert e = fetch_expert(src, j);
        const float wj = w ? w[j] : 1.0f;
        float2 hr[HPL][8];
        bool act[HPL];
#pragma unroll
        for (int m = 0; m < HPL; m++) {
            const int hg = lane + 32 * m;
            act[m] = hg < HG;
#pragma unroll
            for (int i = 0; i < 8; i++) hr[m][i] = make_float2(0.f, 0.f);
            if (act[m]) {
                const float4 *hp = reinterpret_cast<const float4 *>(h + (size_t)j * f + 16 * hg);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    float4 v = hp[i];
                    hr[m][2 * i] = make_float2(v.x, v.y);
                    hr[m][2 * i + 1] = make_float2(v.z, v.w);
                }
            }
        }
        const size_t rowB = (size_t)(f >> 1), rowS = (size_t)(f >> 5);
        for (int c = i0 + s; c < i1; c += U * nsub) {
            uint2 qv[U][HPL];
            uint32_t sv[U][HPL];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int i = c + u * nsub;
#pragma unroll
                for (int m = 0; m < HPL; m++) {
                    const int hg = lane + 32 * m;
                    qv[u][m] = make_uint2(0, 0);
                    sv[u][m] = 255;
                    if (act[m] && i < i1) {
                        qv[u][m] = ld_stream8(e.dp + i * rowB + 8 * (size_t)hg);
                        sv[u][m] = ld_stream_u8(e.ds + i * rowS + (hg >> 1));
                    }
                }
            }
            float v[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < HPL; m++)
                    if (sv[u][m] != 255u) acc += dot16(qv[u][m], hr[m]) * e8m0_scale(sv[u][m]);
                v[u] = acc;
            }
            warp_transpose_reduce<U>(v, lane);
            constexpr int LPV = 32 / U;
            if ((lane % LPV) == 0) {
                const int u = sel_of<U>(lane);
                const int i = c + u * nsub;
                if (i < i1) red[(size_t)j * rows_per_cta + (i - i0)] = v[0] * wj;
            }
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < i1 - i0; t += blockDim.x) {
        float a = 0.f;
        for (int jj = 0; jj < k; jj++) a += red[(size_t)jj * rows_per_cta + t];
        out[i0 + t] = a;
    }
}

// ------------------------------------------------------------- host launch

static int g_num_sms = 0;

int num_sms()
{
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    return g_num_sms;
}

template <typename K>
static int blocks_per_sm(K kernel, int threads, size_t smem)
{
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem) != cudaSuccess ||
        b < 1)
        b = 1;
    return b;
}

constexpr int kU = 4;

// rows kernel: MODE 0 (one matrix) or 1 (gate/up SwiGLU over k experts).
int launch_rows_t1(int mode, const float *x, const ExpertSrc &src, int k, int in, int rows,
                   float *out, cudaStream_t s)
{
    const int G = in / 32;
    const int nwarps = (G + 31) / 32;
    if (nwarps > 16) return K3MOE_EINVAL;
    const int threads = nwarps * 32;
    const long total = (long)k * rows;
    // first guess of the residency to size the per-CTA row range
    const int sms = num_sms();
    int bps = mode ? blocks_per_sm(k3_rows_t1<1, kU>, threads, 0)
                   : blocks_per_sm(k3_rows_t1<0, kU>, threads, 0);
    long target = (long)sms * bps;
    int rpc = (int)((total + target - 1) / target);
    if (rpc < 1) rpc = 1;
    size_t smem = (size_t)nwarps * rpc * 2 * sizeof(float);
    if (smem > 200 * 1024) {
        rpc = (int)(200 * 1024 / ((size_t)nwarps * 2 * sizeof(float)));
        smem = (size_t)nwarps * rpc * 2 * sizeof(float);
    }
    const int grid = (int)((total + rpc - 1) / rpc);
    if (mode) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(k3_rows_t1<1, kU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        k3_rows_t1<1, kU><<<grid, threads, smem, s>>>(x, src, k, in, rows, out, rpc);
    } else {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(k3_rows_t1<0, kU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        k3_rows_t1<0, kU><<<grid, threads, smem, s>>>(x, src, k, in, rows, out, rpc);
    }
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

template <int HPL>
static int launch_down_hpl(const float *h, const ExpertSrc &src, const float *w, int k, int d,
                           int f, float *out, cudaStream_t s)
{
    const int nsub = 16 / k;
    const int threads = k * nsub * 32;
    const int sms = num_sms();
    const int bps = blocks_per_sm(k3_down_t1<HPL, kU>, threads, 0);
    const long target = (long)sms * bps;
    int rpc = (int)((d + target - 1) / target);
    if (rpc < 1) rpc = 1;
    const size_t smem = (size_t)k * rpc * sizeof(float);
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(k3_down_t1<HPL, kU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    const int grid = (d + rpc - 1) / rpc;
    k3_down_t1<HPL, kU><<<grid, threads, smem, s>>>(h, src, w, k, d, f, out, rpc);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int launch_down_t1(const float *h, const ExpertSrc &src, const float *w, int k, int d, int f,
                   float *out, cudaStream_t s)
{
    if (k < 1 || k > 16) return K3MOE_EINVAL;
    const int hpl = (f / 16 + 31) / 32;
    switch (hpl) {
    case 1: return launch_down_hpl<1>(h, src, w, k, d, f, out, s);
    case 2: return launch_down_hpl<2>(h, src, w, k, d, f, out, s);
    case 3: return launch_down_hpl<3>(h, src, w, k, d, f, out, s);
    case 4: return launch_down_hpl<4>(h, src, w, k, d, f, out, s);
    default: return K3MOE_EINVAL;
    }
}

}  // namespace k3
