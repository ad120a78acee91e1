// k3_gemv.cu -- batch-1 MXFP4 expert kernels (sm_103a).
//
//   k3_rows_t1   : gate/up products + SwiGLU for k selected experts (or one
//                  plain matrix, the pages' k3_matmul_mxfp4 primitive)
//   k3_down_t1   : down products of k experts with the weighted combine
//
// Memory-bound design (1.88 weights per byte of HBM traffic):
//   - one lane owns one 32-group of columns for the whole kernel and keeps
//     those 32 activations in registers (as split f16 hi/lo pairs, see
//     k3_device.cuh), so the activation vector is read once per CTA;
//   - a warp reads 512 contiguous bytes of a row per load (16 B per lane,
//     exactly one group), streamed with L1 no-allocate hints; the 32 E8M0
//     bytes of the same groups come in one 32-byte sector;
//   - loads are software-pipelined: the next U rows are in flight while the
//     current U rows are decoded and multiplied;
//   - per-lane partials of U rows are reduced across the warp with a
//     transpose reduction, then across warps in shared memory;
//   - the grid is the SM count times the resident CTAs per SM, with an equal
//     row range per CTA, so every SM streams the same number of bytes.
#include "k3_device.cuh"
#include "k3_launch.cuh"

namespace k3 {

// 32 activations (one group) as two split halves.
struct XGroup {
    XHalf16 a, b;
};

K3_DEV void load_group(const float *x, XGroup &g)
{
    float v[32];
    const float4 *xp = reinterpret_cast<const float4 *>(x);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float4 t = __ldg(xp + i);
        v[4 * i] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
    }
    split16(v, g.a);
    split16(v + 16, g.b);
}

K3_DEV float group_dot(uint4 q, uint32_t e, const XGroup &x)
{
    if (e == 255u) return 0.f;
    const float d = dot16_split(q.x, q.y, x.a) * x.a.inv + dot16_split(q.z, q.w, x.b) * x.b.inv;
    return d * e8m0_scale(e);
}

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
    constexpr int NM = (MODE == 1) ? 2 : 1;
    constexpr int NV = NM * U;

    XGroup xg;
    if (active) {
        load_group(x + 32 * g, xg);
    } else {
        float z[16] = {};
        split16(z, xg.a);
        split16(z, xg.b);
    }

    const long total = (long)k * rows;
    const long q0 = (long)blockIdx.x * rows_per_cta;
    const long q1 = min(q0 + rows_per_cta, total);
    const size_t rowB = (size_t)(in >> 1), rowS = (size_t)G;
    // the row range of a CTA spans at most two experts (rows_per_cta <= rows)
    const int j0 = (int)(q0 / rows);
    const DevExpert e0 = fetch_expert(src, j0);
    const DevExpert e1 = (j0 + 1 < k) ? fetch_expert(src, j0 + 1) : e0;

    uint4 qa[2][U * NM];
    uint32_t sa[2][U * NM];

    auto issue = [&](int buf, long c) {
#pragma unroll
        for (int u = 0; u < U; u++) {
            const long q = c + u;
#pragma unroll
            for (int m = 0; m < NM; m++) {
                qa[buf][u * NM + m] = make_uint4(0, 0, 0, 0);
                sa[buf][u * NM + m] = 255u;
            }
            if (active && q < q1) {
                const int j = (int)(q / rows);
                const int r = (int)(q - (long)j * rows);
                const DevExpert &e = (j == j0) ? e0 : e1;
                qa[buf][u * NM] = ld_stream16(e.gp + r * rowB + 16 * (size_t)g);
                sa[buf][u * NM] = ld_stream_u8(e.gs + r * rowS + g);
                if (MODE == 1) {
                    qa[buf][u * NM + 1] = ld_stream16(e.up + r * rowB + 16 * (size_t)g);
                    sa[buf][u * NM + 1] = ld_stream_u8(e.us + r * rowS + g);
                }
            }
        }
    };
    auto consume = [&](int buf, long c) {
        float v[NV];
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int m = 0; m < NM; m++)
                v[m * U + u] = group_dot(qa[buf][u * NM + m], sa[buf][u * NM + m], xg);
        warp_transpose_reduce<NV>(v, lane);
        constexpr int LPV = 32 / NV;
        if ((lane % LPV) == 0) {
            const int vi = sel_of<NV>(lane);
            const int u = vi % U, which = vi / U;
            const long q = c + u;
            if (q < q1) red[((size_t)warp * rows_per_cta + (q - q0)) * 2 + which] = v[0];
        }
    };

    issue(0, q0);
    for (long c = q0; c < q1; c += 2 * U) {
        if (c + U < q1) issue(1, c + U);
        consume(0, c);
        if (c + 2 * U < q1) issue(0, c + 2 * U);
        if (c + U < q1) consume(1, c + U);
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

// ------------------------------------------------- gate / up, TMA-staged
// Persistent pipeline, one CTA per SM.  The CTA's rows are cut into stages of
// R rows of one expert; a producer lane streams every stage into a ring of S
// shared-memory slots with cp.async.bulk (gate rows, gate scales, up rows, up
// scales: four contiguous copies), arming the slot's `full` mbarrier with the
// byte count.  Compute warps (ncol column slices x RS row sets) read their
// 16-byte group of each row from shared memory, reduce across lanes, and the
// last warp to finish a stage (a per-slot ticket, no waiting) sums the column
// slices in fixed order, applies SwiGLU and writes h.  Then the slot's
// `empty` mbarrier lets the producer refill it.
template <int NM, int R, int RS>
__global__ void __launch_bounds__(512, 1) k3_rows_pipe(const float *__restrict__ x, ExpertSrc src,
                                                       int k, int in, int rows, float *__restrict__ out,
                                                       int nstage_total, int S, int *err)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = in >> 5;
    const int ncol = (G + 31) >> 5;
    const int ncw = ncol * RS;
    const size_t rowB = (size_t)(in >> 1), rowS = (size_t)G;
    const uint32_t matB = (uint32_t)(R * rowB + R * rowS);  // one matrix of one stage
    const uint32_t stageB = NM * matB;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * stageB);     // [S][R][NM][ncol]
    int *cnt = reinterpret_cast<int *>(red + (size_t)S * R * NM * ncol);   // [S]
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        reinterpret_cast<uint8_t *>(cnt) + ((S * sizeof(int) + 7) & ~(size_t)7));  // full[S], empty[S]
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t sbase = smem_u32(smem);

    // this CTA's stages: an equal share of all R-row stages
    const int st0 = (int)(((long)blockIdx.x * nstage_total) / gridDim.x);
    const int st1 = (int)(((long)(blockIdx.x + 1) * nstage_total) / gridDim.x);
    const int nst = st1 - st0;
    const long total = (long)k * rows;

    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, ncw);
            cnt[i] = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == ncw) {  // ------------------------------------------ producer
        // weights of inline experts are requested before the previous
        // kernel on the stream has finished; routed ids are its output
        if (src.ids) griddep_wait();
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < nst && ok; i++) {
                const int slot = i % S;
                if (!mbar_wait(empty0 + 8 * slot, ((i / S) & 1) ^ 1, err)) { ok = false; break; }
                const long q = (long)(st0 + i) * R;
                const int nr = (int)min((long)R, total - q);
                const int j = (int)(q / rows);
                const int r = (int)(q - (long)j * rows);
                const DevExpert e = fetch_expert(src, j);
                const uint32_t dst = sbase + slot * stageB;
                mbar_arrive_expect_tx(full0 + 8 * slot, (uint32_t)(NM * nr * (rowB + rowS)));
                bulk_g2s(dst, e.gp + r * rowB, (uint32_t)(nr * rowB), full0 + 8 * slot);
                bulk_g2s(dst + R * rowB, e.gs + r * rowS, (uint32_t)(nr * rowS), full0 + 8 * slot);
                if (NM == 2) {
                    bulk_g2s(dst + matB, e.up + r * rowB, (uint32_t)(nr * rowB), full0 + 8 * slot);
                    bulk_g2s(dst + matB + R * rowB, e.us + r * rowS, (uint32_t)(nr * rowS),
                             full0 + 8 * slot);
                }
                issued = i + 1;
            }
            if (!ok) {  // consumers are gone: let the copies already issued land
                for (int i = max(0, issued - S); i < issued; i++)
                    mbar_wait(full0 + 8 * (i % S), (i / S) & 1, err);
            }
        }
        return;
    }

    // -------------------------------------------------------------- compute
    griddep_wait();  // x and out belong to the kernels around this one
    const int c = warp % ncol, rs = warp / ncol;
    const int g = c * 32 + lane;
    const bool active = g < G;
    XGroup xg;
    if (active) {
        load_group(x + 32 * g, xg);
    } else {
        float z[16] = {};
        split16(z, xg.a);
        split16(z, xg.b);
    }
    constexpr int NT = R / RS;      // rows of a stage per warp
    constexpr int NV = NT * NM;     // values reduced per stage
    for (int i = 0; i < nst; i++) {
        const int slot = i % S;
        if (!mbar_wait(full0 + 8 * slot, (i / S) & 1, err)) return;
        const long q = (long)(st0 + i) * R;
        const int nr = (int)min((long)R, total - q);
        const uint32_t base = sbase + slot * stageB;
        float v[NV];
#pragma unroll
        for (int t = 0; t < NT; t++) {
            const int row = rs + t * RS;
#pragma unroll
            for (int m = 0; m < NM; m++) {
                float val = 0.f;
                if (active && row < nr) {
                    const uint32_t mb = base + m * matB;
                    const uint4 qv = lds128(mb + row * (uint32_t)rowB + 16 * g);
                    const uint32_t e = lds_u8(mb + R * (uint32_t)rowB + row * (uint32_t)rowS + g);
                    val = group_dot(qv, e, xg);
                }
                v[m * NT + t] = val;
            }
        }
        warp_transpose_reduce<NV>(v, lane);
        constexpr int LPV = 32 / NV;
        if ((lane % LPV) == 0) {
            const int vi = sel_of<NV>(lane);
            const int t = vi % NT, m = vi / NT;
            const int row = rs + t * RS;
            red[(((size_t)slot * R + row) * NM + m) * ncol + c] = v[0];
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = (atomicAdd(&cnt[slot], 1) == ncw - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence_block();
            if (lane < nr) {
                float a = 0.f, b = 0.f;
                for (int cc = 0; cc < ncol; cc++) {
                    a += red[(((size_t)slot * R + lane) * NM + 0) * ncol + cc];
                    if (NM == 2) b += red[(((size_t)slot * R + lane) * NM + 1) * ncol + cc];
                }
                out[q + lane] = (NM == 2) ? silu(a) * b : a;
            }
            if (lane == 0) cnt[slot] = 0;
            __syncwarp();
        }
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    }
}

// -------------------------------------------------------------------- down
// out[i] = sum_j w[j] * (down_j[i] . h[j])  over the k selected experts
// (added to out[i] when acc is set).
// CTA: k * nsub warps; warp (j, s) handles expert j and rows i0+s, i0+s+nsub..
// Lane owns HPL half-groups (16 columns each) of the f-long input.
template <int HPL, int U>
__global__ void __launch_bounds__(512) k3_down_t1(const float *__restrict__ h, ExpertSrc src,
                                                  const float *__restrict__ w, int k, int d, int f,
                                                  float *__restrict__ out, int rows_per_cta,
                                                  int acc)
{
    extern __shared__ float red[];  // [k][rows_per_cta]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nsub = (blockDim.x >> 5) / k;
    const int j = warp % k, s = warp / k;
    const int HG = f >> 4;
    const int i0 = blockIdx.x * rows_per_cta;
    const int i1 = min(i0 + rows_per_cta, d);
    griddep_launch_dependents();
    // routed ids and the combine weights are the previous kernels' output
    if (src.ids) griddep_wait();

    if (s < nsub) {
        const DevExpert e = fetch_expert(src, j);
        float wj = 1.0f;  // the combine weight, read after the wait below
        float2 hr[HPL][8];
        bool act[HPL];
#pragma unroll
        for (int m = 0; m < HPL; m++) {
            act[m] = lane + 32 * m < HG;
#pragma unroll
            for (int i = 0; i < 8; i++) hr[m][i] = make_float2(0.f, 0.f);
        }
        const size_t rowB = (size_t)(f >> 1), rowS = (size_t)(f >> 5);
        uint2 qv[2][U][HPL];
        uint32_t sv[2][U][HPL];
        auto issue = [&](int buf, int c) {
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int i = c + u * nsub;
#pragma unroll
                for (int m = 0; m < HPL; m++) {
                    const int hg = lane + 32 * m;
                    qv[buf][u][m] = make_uint2(0, 0);
                    sv[buf][u][m] = 255u;
                    if (act[m] && i < i1) {
                        qv[buf][u][m] = ld_stream8(e.dp + i * rowB + 8 * (size_t)hg);
                        sv[buf][u][m] = ld_stream_u8(e.ds + i * rowS + (hg >> 1));
                    }
                }
            }
        };
        auto consume = [&](int buf, int c) {
            float v[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < HPL; m++)
                    if (sv[buf][u][m] != 255u)
                        acc += dot16(qv[buf][u][m], hr[m]) * e8m0_scale(sv[buf][u][m]);
                v[u] = acc;
            }
            warp_transpose_reduce<U>(v, lane);
            constexpr int LPV = 32 / U;
            if ((lane % LPV) == 0) {
                const int u = sel_of<U>(lane);
                const int i = c + u * nsub;
                if (i < i1) red[(size_t)j * rows_per_cta + (i - i0)] = v[0] * wj;
            }
        };
        const int step = U * nsub;
        // the first weight rows are requested before h, the previous
        // kernel's output, is read
        issue(0, i0 + s);
        griddep_wait();
        if (w) wj = w[j];
#pragma unroll
        for (int m = 0; m < HPL; m++) {
            if (act[m]) {
                const float4 *hp = reinterpret_cast<const float4 *>(h + (size_t)j * f + 16 * (lane + 32 * m));
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    float4 t = hp[i];
                    hr[m][2 * i] = make_float2(t.x, t.y);
                    hr[m][2 * i + 1] = make_float2(t.z, t.w);
                }
            }
        }
        for (int c = i0 + s; c < i1; c += 2 * step) {
            if (c + step < i1) issue(1, c + step);
            consume(0, c);
            if (c + 2 * step < i1) issue(0, c + 2 * step);
            if (c + step < i1) consume(1, c + step);
        }
    }
    griddep_wait();  // out belongs to the kernels around this one
    __syncthreads();
    for (int t = threadIdx.x; t < i1 - i0; t += blockDim.x) {
        float a = 0.f;
        for (int jj = 0; jj < k; jj++) a += red[(size_t)jj * rows_per_cta + t];
        out[i0 + t] = acc ? out[i0 + t] + a : a;
    }
}

// ------------------------------------------------------------- host launch


template <typename K>
static int blocks_per_sm(K kernel, int threads, size_t smem)
{
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem) != cudaSuccess ||
        b < 1)
        b = 1;
    return b;
}

constexpr int kUrows = 2;  // rows per pipeline stage in the gate/up kernel
constexpr int kUdown = 2;  // rows per pipeline stage in the down kernel

int *device_error_word();

// Pipelined (bulk-copy staged) rows kernel; returns K3MOE_EINVAL when the
// shape does not fit its constraints so the caller can use the direct one.
constexpr int kPipeR = 4;
template <int NM>
static int launch_rows_pipe(const float *x, const ExpertSrc &src, int k, int in, int rows,
                            float *out, int *err, cudaStream_t s)
{
    const int G = in / 32;
    const int ncol = (G + 31) / 32;
    if (in % 128 || rows % kPipeR || ncol > 7) return K3MOE_EINVAL;
    constexpr int RS = 2;
    const int threads = (ncol * RS + 1) * 32;
    const size_t rowB = in / 2, rowS = in / 32;
    const size_t stageB = NM * (kPipeR * rowB + kPipeR * rowS);
    const size_t budget = 200 * 1024;
    int S = 6;
    auto extra = [&](int S_) {
        return (size_t)S_ * kPipeR * NM * ncol * sizeof(float) + ((S_ * sizeof(int) + 7) & ~(size_t)7) +
               2 * S_ * sizeof(uint64_t);
    };
    while (S > 2 && (size_t)S * stageB + extra(S) > budget) S--;
    const size_t smem = (size_t)S * stageB + extra(S);
    if (smem > budget) return K3MOE_EINVAL;
    auto kern = k3_rows_pipe<NM, kPipeR, RS>;
    if (ensure_smem((const void *)kern, smem) != K3MOE_OK) return K3MOE_ECUDA;
    const long total = (long)k * rows;
    const int nstage = (int)((total + kPipeR - 1) / kPipeR);
    int grid = num_sms();
    if (grid > nstage) grid = nstage;
    if (launch_pdl(kern, dim3(grid), dim3(threads), smem, s, x, src, k, in, rows, out, nstage, S, err) !=
        cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ECUDA;
    }
    return K3MOE_OK;
}

// rows kernel: MODE 0 (one matrix) or 1 (gate/up SwiGLU over k experts).
// `err` is the device error word the pipelined kernel reports timeouts to.
int launch_rows_t1_err(int mode, const float *x, const ExpertSrc &src, int k, int in, int rows,
                       float *out, int *err, cudaStream_t s)
{
    {
        const int st = mode ? launch_rows_pipe<2>(x, src, k, in, rows, out, err, s)
                            : launch_rows_pipe<1>(x, src, k, in, rows, out, err, s);
        if (st != K3MOE_EINVAL) return st;
    }
    const int G = in / 32;
    const int nwarps = (G + 31) / 32;
    if (nwarps > 16) return K3MOE_EINVAL;
    const int threads = nwarps * 32;
    const long total = (long)k * rows;
    const int sms = num_sms();
    int bps = mode ? blocks_per_sm(k3_rows_t1<1, kUrows>, threads, 0)
                   : blocks_per_sm(k3_rows_t1<0, kUrows>, threads, 0);
    long target = (long)sms * bps;
    int rpc = (int)((total + target - 1) / target);
    if (rpc < 1) rpc = 1;
    if (rpc > rows) rpc = rows;  // a CTA spans at most two experts
    size_t smem = (size_t)nwarps * rpc * 2 * sizeof(float);
    if (smem > 200 * 1024) {
        rpc = (int)(200 * 1024 / ((size_t)nwarps * 2 * sizeof(float)));
        smem = (size_t)nwarps * rpc * 2 * sizeof(float);
    }
    const int grid = (int)((total + rpc - 1) / rpc);
    if (mode) {
        if (ensure_smem((const void *)k3_rows_t1<1, kUrows>, smem) != K3MOE_OK) return K3MOE_ECUDA;
        k3_rows_t1<1, kUrows><<<grid, threads, smem, s>>>(x, src, k, in, rows, out, rpc);
    } else {
        if (ensure_smem((const void *)k3_rows_t1<0, kUrows>, smem) != K3MOE_OK) return K3MOE_ECUDA;
        k3_rows_t1<0, kUrows><<<grid, threads, smem, s>>>(x, src, k, in, rows, out, rpc);
    }
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int launch_rows_t1(int mode, const float *x, const ExpertSrc &src, int k, int in, int rows,
                   float *out, cudaStream_t s)
{
    return launch_rows_t1_err(mode, x, src, k, in, rows, out, device_error_word(), s);
}

template <int HPL>
static int launch_down_hpl(const float *h, const ExpertSrc &src, const float *w, int k, int d,
                           int f, float *out, cudaStream_t s, bool acc)
{
    const int nsub = 16 / k;
    const int threads = k * nsub * 32;
    const int sms = num_sms();
    const int bps = blocks_per_sm(k3_down_t1<HPL, kUdown>, threads, 0);
    const long target = (long)sms * bps;
    int rpc = (int)((d + target - 1) / target);
    if (rpc < 1) rpc = 1;
    const size_t smem = (size_t)k * rpc * sizeof(float);
    if (ensure_smem((const void *)k3_down_t1<HPL, kUdown>, smem) != K3MOE_OK) return K3MOE_ECUDA;
    const int grid = (d + rpc - 1) / rpc;
    if (launch_pdl(k3_down_t1<HPL, kUdown>, dim3(grid), dim3(threads), smem, s, h, src, w, k, d, f, out, rpc,
                   acc ? 1 : 0) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ECUDA;
    }
    return K3MOE_OK;
}

int launch_down_t1(const float *h, const ExpertSrc &src, const float *w, int k, int d, int f,
                   float *out, cudaStream_t s, bool acc)
{
    if (k < 1 || k > 16) return K3MOE_EINVAL;
    const int hpl = (f / 16 + 31) / 32;
    switch (hpl) {
    case 1: return launch_down_hpl<1>(h, src, w, k, d, f, out, s, acc);
    case 2: return launch_down_hpl<2>(h, src, w, k, d, f, out, s, acc);
    case 3: return launch_down_hpl<3>(h, src, w, k, d, f, out, s, acc);
    case 4: return launch_down_hpl<4>(h, src, w, k, d, f, out, s, acc);
    default: return K3MOE_EINVAL;
    }
}

}  // namespace k3
