// k3_route.cu -- router logits, top-k selection with its combine weights,
// and grouping of (token, slot) pairs by expert (sm_103a).
//
// Router: logits[t][e] = sum_i W_r[e][i] x[t][i], W_r bf16, fp32 accumulate.
// Selection: the top_k largest selection keys (logit + sel_bias, or
// sigmoid(logit) + sel_bias for the sigmoid router), ties to the lower id; the
// combine weights come from the UNBIASED scores of the chosen set ("Running
// Kimi K3 locally", "How is the C engine actually built?", invariant 3).  ids
// are written in ascending order.

#include "k3_device.cuh"

namespace k3 {

int num_sms();


// ------------------------------------------------------- batch-1 router
// The 12.8 MB of W_r for one token are only read at full HBM speed when
// nearly all of them are in flight at once: every expert row is split into S
// column ranges of RT1_CHUNKS 16-byte chunks (S = 4 at d = 7168), one warp
// per (row, range), each lane issuing all its loads (<= RT1_LPL) before the
// first multiply.  Partial dot products go to part[S][E]; the last CTA to
// finish (ticket counter, no waiting) sums them in a fixed order, applies the
// optional RMSNorm factor and runs the top-k.
constexpr int RT1_LPL = 8;                 // 16-byte loads per lane per range
constexpr int RT1_CHUNKS = 32 * RT1_LPL;   // 8-column chunks per range
constexpr int RT1_SMAX = 16;               // ranges per row: d <= 16384

int route_t1_splits(int d) { return ((d >> 3) + RT1_CHUNKS - 1) / RT1_CHUNKS; }

// part: [S][E] partial dot products, then S partial sums of x^2 (RMSNorm
// mode).  RMSNorm mode (u != null, x fp32): r = 1/sqrt(mean(x^2) + eps); the
// logits are r * (W_r . x), equal to W_r . (r x) up to rounding, and u = r x
// is written for the expert kernels.  Otherwise r = 1 and u is not written.
// The last CTA's loads are all issued before their first use (fixed-size
// unrolled loops): a dependent chain of L2 round trips there would cost more
// than the whole matrix read.
template <typename XT>
__global__ void __launch_bounds__(256) k3_router_t1(const XT *__restrict__ x,
                                                    const uint16_t *__restrict__ Wr, int E, int d,
                                                    int S, float *part, float *logits,
                                                    Router rt, int k, int32_t *ids,
                                                    float *w, unsigned *ticket, float eps,
                                                    float *u)
{
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int e = g / S, sp = g - e * S;
    if (e < E) {
        const uint16_t *row = Wr + (size_t)e * d;
        const int c0 = sp * RT1_CHUNKS, c1 = min(c0 + RT1_CHUNKS, d >> 3);
        uint4 wv[RT1_LPL];
#pragma unroll
        for (int q = 0; q < RT1_LPL; q++) {
            const int c = c0 + lane + 32 * q;
            wv[q] = c < c1 ? ld_stream16(row + 8 * c) : make_uint4(0, 0, 0, 0);
        }
        float acc = 0.f, xx = 0.f;
#pragma unroll
        for (int q = 0; q < RT1_LPL; q++) {
            const int c = c0 + lane + 32 * q;
            if (c < c1) {
                float xv[8];
                load_x8<XT>(x, 8 * c, xv);
                acc = bf16x8_dot(wv[q], xv, acc);
#pragma unroll
                for (int i = 0; i < 8; i++) xx = fmaf(xv[i], xv[i], xx);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) part[(size_t)sp * E + e] = acc;
        if (u && e == 0) {  // row 0's S warps cover x once
            xx = warp_sum(xx);
            if (lane == 0) part[(size_t)S * E + sp] = xx;
        }
    }
    __shared__ unsigned s_last;
    __syncthreads();
    if (threadIdx.x == 0) s_last = (ticket_arrive(ticket) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    float r = 1.f;
    if (u) {
        float v[RT1_SMAX];
#pragma unroll
        for (int q = 0; q < RT1_SMAX; q++) v[q] = q < S ? __ldcg(part + (size_t)S * E + q) : 0.f;
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < RT1_SMAX; q++) ss += v[q];
        r = rsqrtf(ss / (float)d + eps);
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        float4 *u4 = reinterpret_cast<float4 *>(u);
        const int n4 = d >> 2;
        for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * blockDim.x) {
            float4 t[8];
#pragma unroll
            for (int q = 0; q < 8; q++) {
                const int i = i0 + q * blockDim.x;
                if (i < n4) t[q] = x4[i];
            }
#pragma unroll
            for (int q = 0; q < 8; q++) {
                const int i = i0 + q * blockDim.x;
                if (i < n4) u4[i] = make_float4(t[q].x * r, t[q].y * r, t[q].z * r, t[q].w * r);
            }
        }
    }
    for (int i0 = threadIdx.x; i0 < E; i0 += 2 * blockDim.x) {
        float v[2][RT1_SMAX];
#pragma unroll
        for (int m = 0; m < 2; m++) {
            const int i = i0 + m * blockDim.x;
#pragma unroll
            for (int q = 0; q < RT1_SMAX; q++)
                v[m][q] = (i < E && q < S) ? __ldcg(part + (size_t)q * E + i) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 2; m++) {
            const int i = i0 + m * blockDim.x;
            float a = 0.f;
#pragma unroll
            for (int q = 0; q < RT1_SMAX; q++) a += v[m][q];
            if (i < E) logits[i] = a * r;
        }
    }
    __syncthreads();
    __shared__ CtaTopkSmem tk;
    cta_topk(logits, rt, E, k, ids, w, tk, [] { __syncthreads(); });
    if (threadIdx.x == 0) *ticket = 0;  // ready for the next launch on this stream
}

// ------------------------------------------------- multi-token router
// Tiled SGEMM: logits[T][E] (split-K partials, summed in fixed order by the
// top-k kernel).  CTA tile: 64 experts x 64 tokens, K step 32, 256 threads,
// each thread 4 x 4 outputs.
constexpr int RT_E = 64, RT_T = 64, RT_K = 32;

template <typename XT>
K3_DEV float to_f(XT v);
template <>
K3_DEV float to_f<float>(float v) { return v; }
template <>
K3_DEV float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename XT>
__global__ void __launch_bounds__(256) k3_router_tiled(const XT *__restrict__ X, int T,
                                                       const uint16_t *__restrict__ Wr, int E,
                                                       int d, int ksplit_len,
                                                       float *__restrict__ part)
{
    __shared__ float sW[RT_K][RT_E + 4];
    __shared__ float sX[RT_K][RT_T + 4];
    const int e0 = blockIdx.x * RT_E, t0 = blockIdx.y * RT_T;
    const int kbeg = blockIdx.z * ksplit_len;
    const int kend = min(kbeg + ksplit_len, d);
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int kk = kbeg; kk < kend; kk += RT_K) {
        for (int idx = threadIdx.x; idx < RT_K * RT_E; idx += 256) {
            const int ee = idx / RT_K, kc = idx % RT_K;
            const int e = e0 + ee, kx = kk + kc;
            float v = 0.f;
            if (e < E && kx < kend) v = __uint_as_float((uint32_t)Wr[(size_t)e * d + kx] << 16);
            sW[kc][ee] = v;
        }
        for (int idx = threadIdx.x; idx < RT_K * RT_T; idx += 256) {
            const int tt = idx / RT_K, kc = idx % RT_K;
            const int t = t0 + tt, kx = kk + kc;
            float v = 0.f;
            if (t < T && kx < kend) v = to_f<XT>(X[(size_t)t * d + kx]);
            sX[kc][tt] = v;
        }
        __syncthreads();
#pragma unroll 8
        for (int kc = 0; kc < RT_K; kc++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = sW[kc][ty * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; i++) b[i] = sX[kc][tx * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int jx = 0; jx < 4; jx++) acc[i][jx] = fmaf(a[i], b[jx], acc[i][jx]);
        }
        __syncthreads();
    }
    float *p = part + (size_t)blockIdx.z * T * E;
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int jx = 0; jx < 4; jx++) {
            const int e = e0 + ty * 4 + i, t = t0 + tx * 4 + jx;
            if (e < E && t < T) p[(size_t)t * E + e] = acc[i][jx];
        }
}

// Sums split-K partials in fixed order, then selects per token (warp/token).
__global__ void __launch_bounds__(256) k3_topk_multi(const float *__restrict__ part, int nsplit,
                                                     int T, int E, Router rt, int k,
                                                     float *logits, int32_t *ids, float *w)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float *lg = logits + (size_t)t * E;
    for (int e = lane; e < E; e += 32) {
        float s = 0.f;
        for (int z = 0; z < nsplit; z++) s += part[((size_t)z * T + t) * E + e];
        lg[e] = s;
    }
    __syncwarp();
    warp_topk(lg, rt, E, k, ids + (size_t)t * k, w + (size_t)t * k, lane);
}

// ---------------------------------------------------------------- grouping
// counts[E] -> offsets[E+1] (exclusive scan) -> perm[pairs] grouped by expert
// (order inside a group is arbitrary; every pair's arithmetic is independent
// of its position) -> a work list of (expert, first pair, n pairs) items of at
// most `nt` pairs each.
__global__ void __launch_bounds__(1024) k3_group(const int32_t *__restrict__ ids, int npairs,
                                                 int E, int nt, int32_t *offsets, int32_t *perm,
                                                 int4 *items, int32_t *n_items)
{
    extern __shared__ int32_t sh[];  // cnt[E], off[E+1], fill[E]
    int32_t *cnt = sh, *off = sh + E, *fill = sh + 2 * E + 1;
    for (int e = threadIdx.x; e < E; e += blockDim.x) { cnt[e] = 0; fill[e] = 0; }
    __syncthreads();
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) atomicAdd(&cnt[ids[p]], 1);
    __syncthreads();
    // offsets and work items by a block-wide exclusive scan over experts
    // (one thread per expert; the layer has at most blockDim experts)
    {
        __shared__ int wsum[2][32];
        const int e = threadIdx.x, lane = e & 31, warp = e >> 5, nw = blockDim.x >> 5;
        const int c = e < E ? cnt[e] : 0, ni = (c + nt - 1) / nt;
        int v[2] = {c, ni}, inc[2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            int x = v[i];
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            inc[i] = x;
            if (lane == 31) wsum[i][warp] = x;
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int i = 0; i < 2; i++) {
                int x = lane < nw ? wsum[i][lane] : 0;
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane < nw) wsum[i][lane] = x - wsum[i][lane];
            }
        }
        __syncthreads();
        const int first = wsum[0][warp] + inc[0] - v[0];   // exclusive prefix of the counts
        const int item0 = wsum[1][warp] + inc[1] - v[1];   // exclusive prefix of the item counts
        if (e < E) {
            off[e] = first;
            for (int b = 0; b < ni; b++) items[item0 + b] = make_int4(e, first + b * nt, min(nt, c - b * nt), 0);
        }
        if (e == blockDim.x - 1) {
            off[E] = first + c;
            *n_items = item0 + ni;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets[e] = off[e];
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
        const int e = ids[p];
        const int slot = atomicAdd(&fill[e], 1);
        perm[off[e] + slot] = p;
    }
}

// ------------------------------------------------------------- launchers

int launch_route_t1(const void *x, int xdt, const uint16_t *Wr, int E, int d, float *part,
                    float *logits, Router rt, int k, int32_t *ids, float *w,
                    unsigned *ticket, float eps, float *u, cudaStream_t s)
{
    const int S = route_t1_splits(d);
    if ((u && xdt != K3MOE_F32) || S > RT1_SMAX) return K3MOE_EINVAL;
    const int threads = 256, wpb = threads / 32;
    const int grid = (int)(((long)E * S + wpb - 1) / wpb);
    if (xdt == K3MOE_F32)
        k3_router_t1<float><<<grid, threads, 0, s>>>((const float *)x, Wr, E, d, S, part, logits,
                                                     rt, k, ids, w, ticket, eps, u);
    else
        k3_router_t1<__nv_bfloat16><<<grid, threads, 0, s>>>((const __nv_bfloat16 *)x, Wr, E, d,
                                                             S, part, logits, rt, k, ids, w,
                                                             ticket, eps, u);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int route_multi_nsplit(int T, int E, int d)
{
    const long tiles = (long)((E + RT_E - 1) / RT_E) * ((T + RT_T - 1) / RT_T);
    long want = (2L * num_sms() + tiles - 1) / tiles;
    int maxs = d / 256;
    if (maxs < 1) maxs = 1;
    if (want > maxs) want = maxs;
    if (want < 1) want = 1;
    return (int)want;
}

int launch_router_tc(const uint16_t *X, int T, const uint16_t *Wr, int E, int d, float *logits, int *err,
                     cudaStream_t s);
int *device_error_word();

int launch_route_multi(const void *X, int xdt, int T, const uint16_t *Wr, int E, int d,
                       float *part, int nsplit, float *logits, Router rt, int k,
                       int32_t *ids, float *w, cudaStream_t s)
{
    // bf16 tokens in numbers: the logits as a tensor-core GEMM
    if (xdt == K3MOE_BF16 && T >= 128 && d % 64 == 0 &&
        launch_router_tc((const uint16_t *)X, T, Wr, E, d, part, device_error_word(), s) == K3MOE_OK) {
        k3_topk_multi<<<(T + 7) / 8, 256, 0, s>>>(part, 1, T, E, rt, k, logits, ids, w);
        return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
    }
    int klen = (d + nsplit - 1) / nsplit;
    klen = (klen + RT_K - 1) / RT_K * RT_K;
    const int ns = (d + klen - 1) / klen;
    dim3 grid((E + RT_E - 1) / RT_E, (T + RT_T - 1) / RT_T, ns);
    if (xdt == K3MOE_F32)
        k3_router_tiled<float><<<grid, 256, 0, s>>>((const float *)X, T, Wr, E, d, klen, part);
    else
        k3_router_tiled<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16 *)X, T, Wr, E,
                                                            d, klen, part);
    k3_topk_multi<<<(T + 7) / 8, 256, 0, s>>>(part, ns, T, E, rt, k, logits, ids, w);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int launch_group(const int32_t *ids, int npairs, int E, int nt, int32_t *offsets, int32_t *perm,
                 int4 *items, int32_t *n_items, cudaStream_t s)
{
    const size_t smem = (size_t)(3 * E + 1) * sizeof(int32_t);
    if (ensure_smem((const void *)k3_group, smem) != K3MOE_OK) return K3MOE_ECUDA;
    k3_group<<<1, 1024, smem, s>>>(ids, npairs, E, nt, offsets, perm, items, n_items);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

}  // namespace k3
