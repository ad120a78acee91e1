// k3_fused.cu -- the whole batch-1 routed-expert layer in one persistent,
// cooperative kernel (one CTA per SM).
//
//   phase R  router logits  (bf16 W_r rows streamed, fp32 x)
//   -- grid barrier (the only one) --
//   phase T  top-k + combine weights (every CTA computes the same selection)
//   phase G  gate/up products + SwiGLU of the k experts -> h   (MXFP4)
//            each finished stage bumps its expert's "h rows done" counter
//   phase D  down products -> w_j * y_j, once its expert's h is complete
//            (waits only on the 1-2 experts this CTA needs); each finished
//            64-row block bumps that block's counter and the k-th arrival
//            sums the k contributions in fixed order: out = sum_j w_j y_j
//
// Weight bytes move global -> shared memory by cp.async.bulk, issued by one
// producer lane into a ring of S slots guarded by full/empty mbarriers.  The
// producer never waits for the compute warps except for ring space: it
// streams the router rows at once, the gate/up rows as soon as this CTA knows
// the selection, and the down rows right after.  A stage is consumed by one
// group of warps that together cover all columns (lane = one 32- or
// 16-column slice); groups take stages in turn and drift independently.  The
// last warp of a group to finish a stage (per-slot ticket) sums the column
// slices in fixed order, so results are deterministic.
//
// Cross-CTA counters are 64-bit and only ever grow: launch number `gen`
// (1, 2, ...) makes the targets gen * grid, gen * (f / 8) and gen * k, so no
// counter is ever reset.  `gen` lives on the device (read at entry, advanced
// by the last CTA to leave), so a captured launch replays correctly.  Every wait is bounded (2 s) and records
// K3MOE_ETIMEOUT in the device error word instead of hanging.
#include "k3_device.cuh"

namespace k3 {

int num_sms();
int *device_error_word();

constexpr int FU_NCW = 14;       // compute warps
constexpr int FU_THREADS = (FU_NCW + 1) * 32;
constexpr int FU_RR = 2;         // router rows per stage
constexpr int FU_RG = 8;         // gate/up rows per stage
constexpr int FU_RD = 64;        // down rows per stage (and combine block)
constexpr int FU_MAXK = 16;
constexpr int FU_REDMAX = 256;   // floats of per-slot reduction buffer
constexpr int FU_CTR_H = 1;      // counters: [0] grid barrier,
constexpr int FU_CTR_Y = 1 + FU_MAXK;  // [1..16] h per expert, [17..] y per block
constexpr int FU_CTR_EXIT = FU_CTR_Y + 7168 / FU_RD;  // CTAs done with this launch
constexpr int FU_CTR_GEN = FU_CTR_EXIT + 1;            // launches completed
constexpr int FU_NCTR = FU_CTR_GEN + 1;

struct FusedArgs {
    const float *x;          // [d]
    const uint16_t *Wr;      // [E][d] bf16
    Router rt;               // selection bias ([E] or null) and score rule
    const DevExpert *table;  // [E]
    int E, k, d, f;
    float *logits;           // [E]
    int32_t *ids;            // [k]  (written by CTA 0)
    float *w;                // [k]  (written by CTA 0)
    float *h;                // [k][f]
    float *Y;                // [k][d]
    float *out;              // [d]
    unsigned long long *ctr; // [FU_NCTR] monotonic counters
    unsigned long long gen;  // launch number, >= 1 (set on the device)
    int *err;
    int S;                   // ring slots
    uint32_t slotB;          // bytes per slot
};

K3_DEV void named_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

K3_DEV unsigned long long ld_acquire64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Spin (bounded) until *p >= target.
K3_DEV bool wait_counter(const unsigned long long *p, unsigned long long target, int *err)
{
    if (ld_acquire64(p) >= target) return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire64(p) < target) {
        __nanosleep(32);
        if (global_ns() - t0 > kWaitLimitNs) {
            set_device_error(err, K3MOE_ETIMEOUT);
            return false;
        }
    }
    return true;
}

// Grid barrier among the compute warps of every CTA (the producer warps do
// not take part).  Returns false when the wait ran out (or had run out).
K3_DEV bool grid_barrier(const FusedArgs &a, int *abort_flag)
{
    named_sync(1, FU_NCW * 32);
    if (threadIdx.x == 0 && *(volatile int *)abort_flag == 0) {
        __threadfence();
        atomicAdd(&a.ctr[0], 1ull);
        if (!wait_counter(&a.ctr[0], a.gen * gridDim.x, a.err)) *abort_flag = 1;
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

// Compute warps 0..7 (named barrier 2): the top k of the scores into sel_ids
// / sel_w (shared memory); CTA 0 also writes them to the layer's ids / w.
K3_DEV void topk_phase(const FusedArgs &a, int *sel_ids, float *sel_w, CtaTopkSmem &tk)
{
    cta_topk(a.logits, a.rt, a.E, a.k, sel_ids, sel_w, tk, [] { named_sync(2, 256); });
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        __syncwarp();
        if (lane < a.k && blockIdx.x == 0) {
            a.ids[lane] = sel_ids[lane];
            a.w[lane] = sel_w[lane];
        }
        __syncwarp();
    }
}

template <bool ACT16>
__global__ void __launch_bounds__(FU_THREADS, 1) k3_moe_t1_fused(FusedArgs a)
{
    a.gen = ld_acquire64(&a.ctr[FU_CTR_GEN]) + 1;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int S = a.S;
    const uint32_t slotB = a.slotB;
    float *red = reinterpret_cast<float *>(smem + (size_t)S * slotB);       // [S][FU_REDMAX]
    int *cnt = reinterpret_cast<int *>(red + (size_t)S * FU_REDMAX);        // [S]
    unsigned *rel = reinterpret_cast<unsigned *>(cnt + S);                  // [S] releases
    int *sel_ids = reinterpret_cast<int *>(rel + S);                        // [FU_MAXK]
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
            mbar_init(empty0 + 8 * i, 1);  // the finishing warp of the consuming group
            cnt[i] = 0;
            rel[i] = 0;
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
    bool dead = false;  // a wait ran out: skip the remaining work, keep the barriers
    // A group takes every ngrp-th stage, so it may come to a slot while the
    // slot still holds an older stage of another group.  Parity waits only
    // tell adjacent phases apart, so first wait until the slot's previous
    // occupant has been released (rel counts releases per slot); then the
    // full barrier is at most one phase away and its parity is unambiguous.
    auto stage_wait = [&](int idx) -> bool {
        if (dead) return false;
        const int slot = idx % S;
        const unsigned need = (unsigned)(idx / S);
        if (*(volatile unsigned *)&rel[slot] < need) {
            const uint64_t t0 = global_ns();
            for (uint32_t n = 1; *(volatile unsigned *)&rel[slot] < need; n++) {
                __nanosleep(20);
                if ((n & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) {
                    set_device_error(a.err, K3MOE_ETIMEOUT);
                    dead = true;
                    *(volatile int *)abort_flag = 1;
                    return false;
                }
            }
        }
        if (!mbar_wait(full0 + 8 * slot, (idx / S) & 1, a.err)) {
            dead = true;
            *(volatile int *)abort_flag = 1;
        }
        return !dead;
    };
    // ticket among the `gsize` warps of a group: true for the last one
    auto ticket = [&](int slot, int gsize) -> bool {
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = (atomicAdd(&cnt[slot], 1) == gsize - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) __threadfence_block();
        return last != 0;
    };
    auto release = [&](int slot) {
        if (lane == 0) {
            cnt[slot] = 0;
            __threadfence_block();
            *(volatile unsigned *)&rel[slot] = *(volatile unsigned *)&rel[slot] + 1u;
            mbar_arrive(empty0 + 8 * slot);
        }
        __syncwarp();
    };
    const int ncolG = d / 1024;                  // warps per group, 32 columns per lane
    const int ngrpG = FU_NCW / ncolG;            // groups in phases R and G
    const int cG = warp % ncolG, grpG = warp / ncolG;
    const bool inG = grpG < ngrpG;
    const int gcol = cG * 32 + lane;             // this lane's group of 32 columns

    // ------------------------------------------------------ phase R: router
    {
        float xv[32];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            float4 t = __ldg(reinterpret_cast<const float4 *>(a.x + 32 * gcol) + q);
            xv[4 * q] = t.x; xv[4 * q + 1] = t.y; xv[4 * q + 2] = t.z; xv[4 * q + 3] = t.w;
        }
        for (int s = inG ? grpG : nR; s < nR; s += ngrpG) {
            const int it = s;
            const int slot = it % S;
            if (!stage_wait(it)) break;
            const int e0 = (r_lo + s) * FU_RR;
            const int nr = min(FU_RR, E - e0);
            for (int row = 0; row < nr; row++) {
                const uint32_t rb = sbase + slot * slotB + row * rRowB + 64 * gcol;
                float acc = 0.f;
#pragma unroll
                for (int q = 0; q < 4; q++) acc = bf16x8_dotf(lds128(rb + 16 * q), xv + 8 * q, acc);
                acc = warp_sum(acc);
                if (lane == 0) red[(size_t)slot * FU_REDMAX + row * ncolG + cG] = acc;
            }
            if (ticket(slot, ncolG)) {
                if (lane < nr) {
                    float sum = 0.f;
                    for (int cc = 0; cc < ncolG; cc++) sum += red[(size_t)slot * FU_REDMAX + lane * ncolG + cc];
                    a.logits[e0 + lane] = sum;
                }
                release(slot);
            }
        }
    }
    if (!grid_barrier(a, abort_flag)) return;

    // ------------------------------------------------------ phase T: top-k
    if (warp < 8) {
        __shared__ CtaTopkSmem tk;
        topk_phase(a, sel_ids, sel_w, tk);
        if (threadIdx.x == 0) {
            __threadfence_block();
            mbar_arrive(topk_bar);  // the producer may now stream expert rows
        }
    }
    named_sync(1, FU_NCW * 32);

    // ------------------------------------------------------ phase G: gate/up
    if (inG) {
        XHalf16 xa, xb;
        {
            float v[32];
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float4 t = __ldg(reinterpret_cast<const float4 *>(a.x + 32 * gcol) + q);
                v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
            }
            split16(v, xa);
            split16(v + 16, xb);
        }
        for (int s = grpG; s < nG; s += ngrpG) {
            const int it = nR + s;
            const int slot = it % S;
            if (!stage_wait(it)) break;
            const int q0 = (g_lo + s) * FU_RG;
            const uint32_t base = sbase + slot * slotB;
#pragma unroll 1
            for (int r0 = 0; r0 < FU_RG; r0 += 4) {  // 4 rows x 2 matrices at a time
                float v[8];                          // [m][row - r0]
#pragma unroll
                for (int t = 0; t < 4; t++) {
#pragma unroll
                    for (int m = 0; m < 2; m++) {
                        const int row = r0 + t;
                        const uint32_t mb = base + m * gMatB;
                        const uint4 qv = lds128(mb + row * (uint32_t)gRowB + 16 * gcol);
                        const uint32_t e = lds_u8(mb + FU_RG * (uint32_t)gRowB + row * (uint32_t)gRowS + gcol);
                        const float dd = dot16_any<ACT16>(qv.x, qv.y, xa) * xa.inv +
                                         dot16_any<ACT16>(qv.z, qv.w, xb) * xb.inv;
                        v[m * 4 + t] = (e == 255u) ? 0.f : dd * e8m0_scale(e);
                    }
                }
                warp_transpose_reduce<8>(v, lane);
                if ((lane & 3) == 0) {
                    const int vi = sel_of<8>(lane);  // m * 4 + t
                    const int m = vi >> 2, row = r0 + (vi & 3);
                    red[(size_t)slot * FU_REDMAX + (m * FU_RG + row) * ncolG + cG] = v[0];
                }
            }
            if (ticket(slot, ncolG)) {
                if (lane < FU_RG) {
                    float gs = 0.f, us = 0.f;
                    for (int cc = 0; cc < ncolG; cc++) {
                        gs += red[(size_t)slot * FU_REDMAX + lane * ncolG + cc];
                        us += red[(size_t)slot * FU_REDMAX + (FU_RG + lane) * ncolG + cc];
                    }
                    a.h[q0 + lane] = silu(gs) * us;
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(&a.ctr[FU_CTR_H + q0 / f], 1ull);  // h rows of expert j done
                }
                release(slot);
            }
        }
    }

    // ------------------------------------------------------ phase D: down
    {
        const int ncolD = f / 512;               // warps per group, 16 columns per lane
        const int ngrpD = FU_NCW / ncolD;
        const int cD = warp % ncolD, grpD = warp / ncolD;
        const int hg = cD * 32 + lane;           // half-group of 16 columns
        if (grpD < ngrpD && nD > 0 && !dead) {
            const int qd0 = d_lo * FU_RD, qd1 = d_hi * FU_RD;
            const int jA = qd0 / d, jB = (qd1 - 1) / d;  // a CTA's share spans <= 2 experts
            const unsigned long long need = a.gen * (unsigned long long)(f / FU_RG);
            bool ok = true;
            if (lane == 0) ok = wait_counter(&a.ctr[FU_CTR_H + jA], need, a.err) &&
                                wait_counter(&a.ctr[FU_CTR_H + jB], need, a.err);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                dead = true;
                *(volatile int *)abort_flag = 1;
            }
            // the group's stages come in expert order: load h_j when j changes
            XHalf16 hx;
            int cur_j = -1;
            for (int s = grpD; s < nD; s += ngrpD) {
                const int it = nR + nG + s;
                const int slot = it % S;
                if (!stage_wait(it)) break;
                const int q0 = (d_lo + s) * FU_RD;
                const int j = q0 / d;
                if (j != cur_j) {
                    float v[16];
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        float4 t = __ldcg(reinterpret_cast<const float4 *>(a.h + (size_t)j * f + 16 * hg) + q);
                        v[4 * q] = t.x; v[4 * q + 1] = t.y; v[4 * q + 2] = t.z; v[4 * q + 3] = t.w;
                    }
                    split16(v, hx);
                    cur_j = j;
                }
                const uint32_t base = sbase + slot * slotB;
                for (int t0 = 0; t0 < FU_RD; t0 += 8) {
                    float v[8];
#pragma unroll
                    for (int t = 0; t < 8; t++) {
                        const int row = t0 + t;
                        const uint2 qv = lds64(base + row * (uint32_t)dRowB + 8 * hg);
                        const uint32_t e = lds_u8(base + FU_RD * (uint32_t)dRowB + row * (uint32_t)dRowS + (hg >> 1));
                        const float dd = dot16_any<ACT16>(qv.x, qv.y, hx) * hx.inv;
                        v[t] = (e == 255u) ? 0.f : dd * e8m0_scale(e);
                    }
                    warp_transpose_reduce<8>(v, lane);
                    if ((lane & 3) == 0) {
                        const int t = sel_of<8>(lane);
                        red[(size_t)slot * FU_REDMAX + (t0 + t) * ncolD + cD] = v[0];
                    }
                }
                if (ticket(slot, ncolD)) {
                    const float wj = sel_w[j];
                    for (int row = lane; row < FU_RD; row += 32) {
                        float sum = 0.f;
                        for (int cc = 0; cc < ncolD; cc++) sum += red[(size_t)slot * FU_REDMAX + row * ncolD + cc];
                        a.Y[q0 + row] = sum * wj;
                    }
                    release(slot);
                    // combine this 64-row block once all k experts wrote it
                    const int blk = (q0 - j * d) / FU_RD;
                    unsigned long long old = 0;
                    if (lane == 0) {
                        __threadfence();
                        old = atomicAdd(&a.ctr[FU_CTR_Y + blk], 1ull);
                    }
                    old = __shfl_sync(0xffffffffu, old, 0);
                    if (old + 1 == a.gen * (unsigned long long)k) {
                        __threadfence();
                        const int i0 = blk * FU_RD;
                        for (int row = lane; row < FU_RD; row += 32) {
                            float acc = 0.f;
                            for (int jj = 0; jj < k; jj++) acc += __ldcg(a.Y + (size_t)jj * d + i0 + row);
                            a.out[i0 + row] = acc;
                        }
                    }
                }
            }
        }
    }
    // the last CTA to leave advances the launch number
    named_sync(1, FU_NCW * 32);
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned long long old = atomicAdd(&a.ctr[FU_CTR_EXIT], 1ull);
        if (old + 1 == a.gen * (unsigned long long)gridDim.x) atomicAdd(&a.ctr[FU_CTR_GEN], 1ull);
    }
}

// ------------------------------------------------------------------- host

// Whether the fused kernel supports this shape.
bool fused_t1_supported(int E, int k, int d, int f)
{
    return d % 1024 == 0 && d >= 1024 && d <= 7168 && f % 512 == 0 && f >= 512 && f <= 2048 &&
           k >= 1 && k <= FU_MAXK && E >= k && E <= 1024 && (k * f) % FU_RG == 0 &&
           d % FU_RD == 0;
}

int fused_t1_counters() { return FU_NCTR; }

size_t fused_t1_smem(int d, int f, int *S_out, uint32_t *slot_out)
{
    const size_t rB = (size_t)FU_RR * d * 2;
    const size_t gB = 2 * (size_t)FU_RG * (d / 2 + d / 32);
    const size_t dB = (size_t)FU_RD * (f / 2 + f / 32);
    size_t slot = rB > gB ? rB : gB;
    if (dB > slot) slot = dB;
    slot = (slot + 127) & ~(size_t)127;
    int S = 8;
    auto total = [&](int s) {
        return (size_t)s * slot + (size_t)s * FU_REDMAX * 4 + (size_t)s * 8 + FU_MAXK * 8 + 4 + 8 +
               (2 * s + 1) * 8;
    };
    while (S > 2 && total(S) > 220 * 1024) S--;
    *S_out = S;
    *slot_out = (uint32_t)slot;
    return total(S);
}

int launch_fused_t1(const float *x, const uint16_t *Wr, Router rt, const DevExpert *table,
                    int E, int k, int d, int f, float *logits, int32_t *ids, float *w, float *h,
                    float *Y, float *out, unsigned long long *ctr, bool act16, cudaStream_t s)
{
    FusedArgs a;
    a.x = x;
    a.Wr = Wr;
    a.rt = rt;
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
    a.ctr = ctr;
    a.gen = 0;
    a.err = device_error_word();
    int S = 0;
    uint32_t slot = 0;
    const size_t smem = fused_t1_smem(d, f, &S, &slot);
    a.S = S;
    a.slotB = slot;
    auto kern = act16 ? k3_moe_t1_fused<true> : k3_moe_t1_fused<false>;
    // one CTA per SM must fit (the grid barrier needs every CTA resident;
    // the cooperative launch refuses a grid that does not)
    if (ensure_smem((const void *)kern, smem) != K3MOE_OK) return K3MOE_ECUDA;
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
