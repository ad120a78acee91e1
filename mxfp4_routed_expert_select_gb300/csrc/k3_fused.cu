// k3_fused.cu -- the whole batch-1 routed-expert layer in one persistent,
// cooperative kernel (one CTA per SM).
//
//   phase R  router logits  (bf16 W_r rows streamed, fp32 x)
//   -- grid barrier --
//   phase T  top-k + softmax (every CTA computes the same selection)
//   phase G  gate/up products + SwiGLU of the k experts -> h   (MXFP4)
//   -- grid barrier --
//   phase D  down products -> w_j * y_j                          (MXFP4)
//   -- grid barrier --
//   phase C  combine: out[i] = sum_j w_j y_j[i]  (fixed order)
//
// Weight bytes move global -> shared memory by cp.async.bulk, issued by one
// producer lane into a ring of S slots guarded by full/empty mbarriers.  The
// producer never takes part in the grid barriers: it streams the router rows
// at once, the gate/up rows as soon as this CTA knows the selection, and the
// down rows right after, so the down weights are already arriving while the
// compute warps wait at the second grid barrier.  Fourteen compute warps read
// their column slice of each staged row from shared memory and decode E2M1 in
// registers (k3_device.cuh, split-activation form).  The last warp to finish a
// stage (per-slot ticket) sums the column slices in fixed order, so results
// are deterministic.  Every wait is bounded (2 s) and records K3MOE_ETIMEOUT
// in the device error word instead of hanging.
#include "k3_device.cuh"

namespace k3 {

int num_sms();
int *device_error_word();

constexpr int FU_NCW = 14;       // compute warps
constexpr int FU_THREADS = (FU_NCW + 1) * 32;
constexpr int FU_RR = 2;         // router rows per stage
constexpr int FU_RG = 8;         // gate/up rows per stage
constexpr int FU_RD = 64;        // down rows per stage
constexpr int FU_MAXK = 16;
constexpr int FU_REDMAX = 256;   // floats of per-slot reduction buffer

struct FusedArgs {
    const float *x;          // [d]
    const uint16_t *Wr;      // [E][d] bf16
    const float *bias;       // [E] or null
    const DevExpert *table;  // [E]
    int E, k, d, f;
    float *logits;           // [E]
    int32_t *ids;            // [k]  (written by CTA 0)
    float *w;                // [k]  (written by CTA 0)
    float *h;                // [k][f]
    float *Y;                // [k][d]
    float *out;              // [d]
    unsigned *gbar;          // [2] arrivals, exits
    int *err;
    int S;                   // ring slots
    uint32_t slotB;          // bytes per slot
};

K3_DEV void named_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

K3_DEV unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier among the compute warps of every CTA (the producer warps do
// not take part).  Returns false when the wait ran out.
K3_DEV bool grid_barrier(const FusedArgs &a, unsigned target, int *abort_flag)
{
    named_sync(1, FU_NCW * 32);
    if (threadIdx.x == 0 && *(volatile int *)abort_flag == 0) {
        __threadfence();
        atomicAdd(&a.gbar[0], 1u);
        const uint64_t t0 = global_ns();
        while (ld_acquire(&a.gbar[0]) < target) {
            __nanosleep(64);
            if (global_ns() - t0 > kWaitLimitNs) {
                set_device_error(a.err, K3MOE_ETIMEOUT);
                *abort_flag = 1;
                break;
            }
        }
        __threadfence();
    }
    named_sync(1, FU_NCW * 32);
    return *(volatile int *)abort_flag == 0;
}

// equal share [lo, hi) of n items for CTA b of nb
K3_DEV void share(int n, int b, int nb, int &lo, int &hi)
{
    lo = (int)(((long)b * n) / nb);
    hi = (int)(((long)(b + 1) * n) / nb);
}

K3_DEV float bf16x8_dotf(uint4 wv, const float *xv, float acc)
{
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        acc = fmaf(__uint_as_float(w[q] << 16), xv[2 * q], acc);
        acc = fmaf(__uint_as_float(w[q] & 0xffff0000u), xv[2 * q + 1], acc);
    }
    return acc;
}

K3_DEV bool fu_better(float a, int ia, float b, int ib) { return a > b || (a == b && ia < ib); }

template <bool ACT16>
__global__ void __launch_bounds__(FU_THREADS, 1) k3_moe_t1_fused(FusedArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = a.S;
    const uint32_t slotB = a.slotB;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * slotB);       // [S][FU_REDMAX]
    int *cnt = reinterpret_cast<int *>(red + (size_t)S * FU_REDMAX);        // [S]
    int *sel_ids = cnt + S;                                                 // [FU_MAXK]
    float *sel_w = reinterpret_cast<float *>(sel_ids + FU_MAXK);            // [FU_MAXK]
    int *abort_flag = reinterpret_cast<int *>(sel_w + FU_MAXK);             // [1]
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(abort_flag + 1) + 7) & ~(uintptr_t)7);  // full[S], empty[S], topk
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t topk_bar = smem_u32(bars + 2 * S);
    const uint32_t sbase = smem_u32(smem);

    const int d = a.d, f = a.f, k = a.k, E = a.E;
    const size_t gRowB = (size_t)(d >> 1), gRowS = (size_t)(d >> 5);   // gate/up rows
    const size_t dRowB = (size_t)(f >> 1), dRowS = (size_t)(f >> 5);   // down rows
    const uint32_t gMatB = (uint32_t)(FU_RG * (gRowB + gRowS));         // one matrix, one stage
    const uint32_t rRowB = (uint32_t)(d * 2);                            // router row bytes

    // this CTA's shares of the three streams (in stages)
    int r_lo, r_hi, g_lo, g_hi, d_lo, d_hi;
    share((E + FU_RR - 1) / FU_RR, blockIdx.x, gridDim.x, r_lo, r_hi);
    share(k * f / FU_RG, blockIdx.x, gridDim.x, g_lo, g_hi);
    share(k * d / FU_RD, blockIdx.x, gridDim.x, d_lo, d_hi);
    const int nR = r_hi - r_lo, nG = g_hi - g_lo, nD = d_hi - d_lo;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, FU_NCW);
            cnt[i] = 0;
        }
        mbar_init(topk_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // ================================================================ producer
    if (warp == FU_NCW) {
        if (lane != 0) return;
        int i = 0;  // global stage index (ring position)
        bool ok = true;
        auto slot_ready = [&](int idx) -> int {
            const int slot = idx % S;
            if (!mbar_wait(empty0 + 8 * slot, ((idx / S) & 1) ^ 1, a.err)) ok = false;
            return slot;
        };
        for (int s = 0; s < nR && ok; s++, i++) {
            const int slot = slot_ready(i);
            if (!ok) break;
            const int e0 = (r_lo + s) * FU_RR;
            const int nr = min(FU_RR, E - e0);
            mbar_arrive_expect_tx(full0 + 8 * slot, nr * rRowB);
            bulk_g2s(sbase + slot * slotB, a.Wr + (size_t)e0 * d, nr * rRowB, full0 + 8 * slot);
        }
        // the selection is needed for every expert stage
        if (ok && !mbar_wait(topk_bar, 0, a.err)) ok = false;
        for (int s = 0; s < nG && ok; s++, i++) {
            const int slot = slot_ready(i);
            if (!ok) break;
            const int q = (g_lo + s) * FU_RG;
            const int j = q / f, r = q - j * f;
            const DevExpert e = a.table[sel_ids[j]];
            const uint32_t dst = sbase + slot * slotB, fb = full0 + 8 * slot;
            mbar_arrive_expect_tx(fb, 2u * FU_RG * (uint32_t)(gRowB + gRowS));
            bulk_g2s(dst, e.gp + r * gRowB, FU_RG * (uint32_t)gRowB, fb);
            bulk_g2s(dst + FU_RG * gRowB, e.gs + r * gRowS, FU_RG * (uint32_t)gRowS, fb);
            bulk_g2s(dst + gMatB, e.up + r * gRowB, FU_RG * (uint32_t)gRowB, fb);
            bulk_g2s(dst + gMatB + FU_RG * gRowB, e.us + r * gRowS, FU_RG * (uint32_t)gRowS, fb);
        }
        for (int s = 0; s < nD && ok; s++, i++) {
            const int slot = slot_ready(i);
            if (!ok) break;
            const int q = (d_lo + s) * FU_RD;
            const int j = q / d, r = q - j * d;
            const DevExpert e = a.table[sel_ids[j]];
            const uint32_t dst = sbase + slot * slotB, fb = full0 + 8 * slot;
            mbar_arrive_expect_tx(fb, FU_RD * (uint32_t)(dRowB + dRowS));
            bulk_g2s(dst, e.dp + r * dRowB, FU_RD * (uint32_t)dRowB, fb);
            bulk_g2s(dst + FU_RD * dRowB, e.ds + r * dRowS, FU_RD * (uint32_t)dRowS, fb);
        }
        if (!ok) {  // consumers gone: let the copies already issued land
            for (int q = max(0, i - S); q < i; q++) mbar_wait(full0 + 8 * (q % S), (q / S) & 1, a.err);
        }
        return;
    }

    // ============================================================ compute warps
    int it = 0;  // ring position, in step with the producer
    unsigned gen = 0;
    auto stage_wait = [&](int idx) -> bool {
        return mbar_wait(full0 + 8 * (idx % S), (idx / S) & 1, a.err);
    };
    // ticket: returns true for the last of the FU_NCW warps on this slot
    auto ticket = [&](int slot) -> bool {
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = (atomicAdd(&cnt[slot], 1) == FU_NCW - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) __threadfence_block();
        return last != 0;
    };
    auto release = [&](int slot, bool last) {
        if (last && lane == 0) cnt[slot] = 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    };

    // ------------------------------------------------------ phase R: router
    {
        const int ncol = d / 1024;              // 32 columns per lane
        const int rs_n = FU_NCW / ncol;
        const int c = warp % ncol, rs = warp / ncol;
        const bool wact = warp < ncol * rs_n;
        const int g = c * 32 + lane;             // group of 32 columns
        float xv[32];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            float4 t = __ldg(reinterpret_cast<const float4 *>(a.x + 32 * g) + q);
            xv[4 * q] = t.x; xv[4 * q + 1] = t.y; xv[4 * q + 2] = t.z; xv[4 * q + 3] = t.w;
        }
        for (int s = 0; s < nR; s++, it++) {
            const int slot = it % S;
            if (!stage_wait(it)) { *(volatile int *)abort_flag = 1; break; }
            const int e0 = (r_lo + s) * FU_RR;
            const int nr = min(FU_RR, E - e0);
            if (wact) {
                for (int row = rs; row < nr; row += rs_n) {
                    const uint32_t rb = sbase + slot * slotB + row * rRowB + 64 * g;
                    float acc = 0.f;
#pragma unroll
                    for (int q = 0; q < 4; q++) acc = bf16x8_dotf(lds128(rb + 16 * q), xv + 8 * q, acc);
                    acc = warp_sum(acc);
                    if (lane == 0) red[(size_t)slot * FU_REDMAX + row * ncol + c] = acc;
                }
            }
            const bool last = ticket(slot);
            if (last && lane < nr) {
                float sum = 0.f;
                for (int cc = 0; cc < ncol; cc++) sum += red[(size_t)slot * FU_REDMAX + lane * ncol + cc];
                a.logits[e0 + lane] = sum;
            }
            release(slot, last);
        }
    }
    if (!grid_barrier(a, gridDim.x * (++gen), abort_flag)) return;

    // ------------------------------------------------------ phase T: top-k
    // Two levels: every compute warp selects the top k of its slice of the
    // E scores (scores in registers, k rounds of a warp argmax), writes the k
    // candidates to shared memory; warp 0 then selects the top k of the
    // FU_NCW * k candidates.  Order: larger score first, ties to lower id.
    {
        float *cand_s = red;                                                  // [FU_NCW][FU_MAXK]
        int *cand_i = reinterpret_cast<int *>(red + FU_NCW * FU_MAXK);       // [FU_NCW][FU_MAXK]
        const int per = (E + FU_NCW - 1) / FU_NCW;                           // slice length <= 74
        const int e_lo = warp * per;
        float sc[3];
        int si[3];
#pragma unroll
        for (int q = 0; q < 3; q++) {
            const int e = e_lo + lane + 32 * q;
            const bool in = (lane + 32 * q < per) && e < E;
            sc[q] = in ? __ldcg(a.logits + e) + (a.bias ? __ldg(a.bias + e) : 0.f) : -INFINITY;
            si[q] = in ? e : 0x7fffffff;
        }
        for (int r = 0; r < k; r++) {
            float bs = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int q = 0; q < 3; q++)
                if (fu_better(sc[q], si[q], bs, bi)) { bs = sc[q]; bi = si[q]; }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (fu_better(os, oi, bs, bi)) { bs = os; bi = oi; }
            }
#pragma unroll
            for (int q = 0; q < 3; q++)
                if (si[q] == bi) { sc[q] = -INFINITY; si[q] = 0x7fffffff; }
            if (lane == 0) {
                cand_s[warp * FU_MAXK + r] = bs;
                cand_i[warp * FU_MAXK + r] = bi;
            }
        }
        named_sync(1, FU_NCW * 32);
        if (warp == 0) {
            constexpr int NC = (FU_NCW * FU_MAXK + 31) / 32;  // candidates per lane
            float cs[NC];
            int ci[NC];
#pragma unroll
            for (int q = 0; q < NC; q++) {
                const int c = lane + 32 * q;
                const bool in = c < FU_NCW * FU_MAXK && (c % FU_MAXK) < k;
                cs[q] = in ? cand_s[c] : -INFINITY;
                ci[q] = in ? cand_i[c] : 0x7fffffff;
            }
            int my_id = -1;
            for (int r = 0; r < k; r++) {
                float bs = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int q = 0; q < NC; q++)
                    if (fu_better(cs[q], ci[q], bs, bi)) { bs = cs[q]; bi = ci[q]; }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) {
                    const float os = __shfl_xor_sync(0xffffffffu, bs, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (fu_better(os, oi, bs, bi)) { bs = os; bi = oi; }
                }
#pragma unroll
                for (int q = 0; q < NC; q++)
                    if (ci[q] == bi) { cs[q] = -INFINITY; ci[q] = 0x7fffffff; }
                if (lane == r) my_id = bi;
            }
            int pos = 0;
            for (int q = 0; q < k; q++) {
                const int other = __shfl_sync(0xffffffffu, my_id, q);
                if (lane < k && other < my_id) pos++;
            }
            const float l = (lane < k) ? __ldcg(a.logits + my_id) : -INFINITY;
            float mx = l;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float ex = (lane < k) ? expf(l - mx) : 0.f;
            const float sum = warp_sum(ex);
            if (lane < k) {
                sel_ids[pos] = my_id;
                sel_w[pos] = ex / sum;
                if (blockIdx.x == 0) {
                    a.ids[pos] = my_id;
                    a.w[pos] = ex / sum;
                }
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                mbar_arrive(topk_bar);  // the producer may now stream expert rows
            }
        }
        named_sync(1, FU_NCW * 32);
    }

    // ------------------------------------------------------ phase G: gate/up
    {
        const int ncol = d / 1024;
        const int rs_n = FU_NCW / ncol;
        const int c = warp % ncol, rs = warp / ncol;
        const bool wact = warp < ncol * rs_n;
        const int g = c * 32 + lane;
        XHalf16 xa, xb;
        {
            float v[32];
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float4 t = __ldg(reinterpret_cast<const float4 *>(a.x + 32 * g) + q);
                v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
            }
            split16(v, xa);
            split16(v + 16, xb);
        }
        constexpr int NT = 4;  // rows per warp per stage (FU_RG / 2 row sets at most)
        for (int s = 0; s < nG; s++, it++) {
            const int slot = it % S;
            if (!stage_wait(it)) { *(volatile int *)abort_flag = 1; break; }
            const int q0 = (g_lo + s) * FU_RG;
            if (wact) {
                const uint32_t base = sbase + slot * slotB;
                // rows rs, rs + rs_n, ... of the stage (at most NT per warp)
                float v[2 * NT];
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const int row = rs + t * rs_n;
#pragma unroll
                    for (int m = 0; m < 2; m++) {
                        float val = 0.f;
                        if (row < FU_RG) {
                            const uint32_t mb = base + m * gMatB;
                            const uint4 qv = lds128(mb + row * (uint32_t)gRowB + 16 * g);
                            const uint32_t e = lds_u8(mb + FU_RG * (uint32_t)gRowB + row * (uint32_t)gRowS + g);
                            const float dd = dot16_any<ACT16>(qv.x, qv.y, xa) * xa.inv +
                                             dot16_any<ACT16>(qv.z, qv.w, xb) * xb.inv;
                            val = (e == 255u) ? 0.f : dd * e8m0_scale(e);
                        }
                        v[m * NT + t] = val;
                    }
                }
                warp_transpose_reduce<2 * NT>(v, lane);
                constexpr int LPV = 32 / (2 * NT);
                if ((lane % LPV) == 0) {
                    const int vi = sel_of<2 * NT>(lane);
                    const int t = vi % NT, m = vi / NT;
                    const int row = rs + t * rs_n;
                    if (row < FU_RG) red[(size_t)slot * FU_REDMAX + (row * 2 + m) * ncol + c] = v[0];
                }
            }
            const bool last = ticket(slot);
            if (last && lane < FU_RG) {
                float gs = 0.f, us = 0.f;
                for (int cc = 0; cc < ncol; cc++) {
                    gs += red[(size_t)slot * FU_REDMAX + (lane * 2 + 0) * ncol + cc];
                    us += red[(size_t)slot * FU_REDMAX + (lane * 2 + 1) * ncol + cc];
                }
                a.h[q0 + lane] = silu(gs) * us;
            }
            release(slot, last);
        }
    }
    if (!grid_barrier(a, gridDim.x * (++gen), abort_flag)) return;

    // ------------------------------------------------------ phase D: down
    {
        const int ncol = f / 512;                // 16 columns per lane
        const int rs_n = FU_NCW / ncol;
        const int c = warp % ncol, rs = warp / ncol;
        const bool wact = warp < ncol * rs_n;
        const int hg = c * 32 + lane;            // half-group of 16 columns
        const int qd0 = d_lo * FU_RD, qd1 = d_hi * FU_RD;
        const int jA = (nD > 0) ? qd0 / d : 0;
        const int jB = (nD > 0) ? (qd1 - 1) / d : 0;  // a CTA's share spans <= 2 experts
        XHalf16 hA, hB;
        {
            float v[16];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float4 t = __ldcg(reinterpret_cast<const float4 *>(a.h + (size_t)jA * f + 16 * hg) + q);
                v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
            }
            split16(v, hA);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float4 t = __ldcg(reinterpret_cast<const float4 *>(a.h + (size_t)jB * f + 16 * hg) + q);
                v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
            }
            split16(v, hB);
        }
        for (int s = 0; s < nD; s++, it++) {
            const int slot = it % S;
            if (!stage_wait(it)) { *(volatile int *)abort_flag = 1; break; }
            const int q0 = (d_lo + s) * FU_RD;
            const int j = q0 / d;
            if (wact) {
                XHalf16 hx;
                const bool useA = (j == jA);
#pragma unroll
                for (int q = 0; q < 16; q++) {
                    hx.hi[q] = useA ? hA.hi[q] : hB.hi[q];
                    hx.lo[q] = useA ? hA.lo[q] : hB.lo[q];
                }
                hx.inv = useA ? hA.inv : hB.inv;
                const uint32_t base = sbase + slot * slotB;
                for (int t0 = 0; rs + t0 * rs_n < FU_RD; t0 += 8) {
                    float v[8];
#pragma unroll
                    for (int t = 0; t < 8; t++) {
                        const int row = rs + (t0 + t) * rs_n;
                        float val = 0.f;
                        if (row < FU_RD) {
                            const uint2 qv = lds64(base + row * (uint32_t)dRowB + 8 * hg);
                            const uint32_t e = lds_u8(base + FU_RD * (uint32_t)dRowB + row * (uint32_t)dRowS + (hg >> 1));
                            const float dd = dot16_any<ACT16>(qv.x, qv.y, hx) * hx.inv;
                            val = (e == 255u) ? 0.f : dd * e8m0_scale(e);
                        }
                        v[t] = val;
                    }
                    warp_transpose_reduce<8>(v, lane);
                    if ((lane & 3) == 0) {
                        const int t = sel_of<8>(lane);
                        const int row = rs + (t0 + t) * rs_n;
                        if (row < FU_RD) red[(size_t)slot * FU_REDMAX + row * ncol + c] = v[0];
                    }
                }
            }
            const bool last = ticket(slot);
            if (last) {
                const float wj = sel_w[j];
                for (int row = lane; row < FU_RD; row += 32) {
                    float sum = 0.f;
                    for (int cc = 0; cc < ncol; cc++) sum += red[(size_t)slot * FU_REDMAX + row * ncol + cc];
                    a.Y[q0 + row] = sum * wj;
                }
            }
            release(slot, last);
        }
    }
    if (!grid_barrier(a, gridDim.x * (++gen), abort_flag)) return;

    // ------------------------------------------------------ phase C: combine
    {
        int i_lo, i_hi;
        share(d, blockIdx.x, gridDim.x, i_lo, i_hi);
        for (int i = i_lo + threadIdx.x; i < i_hi; i += FU_NCW * 32) {
            float acc = 0.f;
            for (int j = 0; j < k; j++) acc += __ldcg(a.Y + (size_t)j * d + i);
            a.out[i] = acc;
        }
    }
    // the last CTA out resets the barrier counters for the next launch
    named_sync(1, FU_NCW * 32);
    if (threadIdx.x == 0) {
        const unsigned old = atomicAdd(&a.gbar[1], 1u);
        if (old == gridDim.x - 1) {
            atomicExch(&a.gbar[0], 0u);
            atomicExch(&a.gbar[1], 0u);
        }
    }
}

// ------------------------------------------------------------------- host

// Whether the fused kernel supports this shape.
bool fused_t1_supported(int E, int k, int d, int f)
{
    return d % 1024 == 0 && d >= 1024 && d <= 7168 && f % 512 == 0 && f >= 512 && f <= 2048 &&
           k >= 1 && k <= FU_MAXK && E >= k && E <= 1024 && (k * f) % FU_RG == 0 &&
           (k * d) % FU_RD == 0 && FU_RD * (f / 2) + FU_RD * (f / 32) > 0;
}

size_t fused_t1_smem(int d, int f, int *S_out, uint32_t *slot_out)
{
    const size_t rB = (size_t)FU_RR * d * 2;
    const size_t gB = 2 * (size_t)FU_RG * (d / 2 + d / 32);
    const size_t dB = (size_t)FU_RD * (f / 2 + f / 32);
    size_t slot = rB > gB ? rB : gB;
    if (dB > slot) slot = dB;
    slot = (slot + 127) & ~(size_t)127;
    const size_t tail = 0;
    int S = 8;
    auto total = [&](int s) {
        return (size_t)s * slot + (size_t)s * FU_REDMAX * 4 + (size_t)s * 4 + FU_MAXK * 8 + 4 + 8 +
               (2 * s + 1) * 8 + tail;
    };
    while (S > 2 && total(S) > 220 * 1024) S--;
    *S_out = S;
    *slot_out = (uint32_t)slot;
    return total(S);
}

int launch_fused_t1(const float *x, const uint16_t *Wr, const float *bias, const DevExpert *table,
                    int E, int k, int d, int f, float *logits, int32_t *ids, float *w, float *h,
                    float *Y, float *out, unsigned *gbar, bool act16, cudaStream_t s)
{
    FusedArgs a;
    a.x = x;
    a.Wr = Wr;
    a.bias = bias;
    a.table = table;
    a.E = E;
    a.k = k;
    a.d = d;
    a.f = f;
    a.logits = logits;
    a.ids = ids;
    a.w = w;
    a.h = h;
    a.Y = Y;
    a.out = out;
    a.gbar = gbar;
    a.err = device_error_word();
    int S = 0;
    uint32_t slot = 0;
    const size_t smem = fused_t1_smem(d, f, &S, &slot);
    a.S = S;
    a.slotB = slot;
    auto kern = act16 ? k3_moe_t1_fused<true> : k3_moe_t1_fused<false>;
    static size_t configured[2] = {0, 0};
    if (smem > configured[act16]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return K3MOE_ECUDA;
        configured[act16] = smem;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, FU_THREADS, smem) != cudaSuccess ||
        per_sm < 1)
        return K3MOE_ECUDA;
    const int grid = num_sms();  // one CTA per SM, all co-resident
    void *args[] = {&a};
    if (cudaLaunchCooperativeKernel((const void *)kern, dim3(grid), dim3(FU_THREADS), args, smem, s) !=
        cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ECUDA;
    }
    return K3MOE_OK;
}

}  // namespace k3
