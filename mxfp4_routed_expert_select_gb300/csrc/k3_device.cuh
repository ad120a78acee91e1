// k3_device.cuh -- device helpers shared by the k3moe kernels (sm_103a).
//
// MXFP4 decode in registers: one byte holds two 4-bit E2M1 codes, the low
// nibble being the even-index weight ("Running Kimi K3 locally", four
// reductions).  The hardware conversion cvt.rn.f16x2.e2m1x2 turns one byte
// into an f16x2 pair (low nibble -> low half); every E2M1 value is exact in
// f16, so the pair converts exactly to two fp32 values.  Products and sums are
// fp32 (packed FFMA2).  The per-32 E8M0 scale is applied once per group, after
// the group's dot product ("kimi-k3-in-c" explainer, "Reduction one").
#pragma once
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "k3moe.h"

#define K3_DEV __device__ __forceinline__

namespace k3 {

// Per-device host state (k3_runtime.cu): the device error word's address,
// the SM count, and a kernel's dynamic shared-memory limit raised to `bytes`.
int *device_error_word();
int num_sms();
int ensure_smem(const void *fn, size_t bytes);

// Programmatic dependent launch: a kernel launched as a dependent of the
// previous one on its stream may start while that one still runs; before it
// reads anything that kernel writes (or writes anything it reads) it waits
// here until that kernel has completed and its memory is visible.  Both are
// no-ops for a kernel launched without the attribute.
K3_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
K3_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Device error word (bounded waits that ran out write K3MOE_ETIMEOUT here):
// one int per device, a file-scope device variable (k3::device_error_word()).
K3_DEV void set_device_error(int *err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

// Device-side expert view: the six plane pointers of one expert.
struct DevExpert {
    const uint8_t *gp, *gs, *up, *us, *dp, *ds;
};

// Where a kernel finds the expert of selection slot j: either a device table
// indexed by device ids, or an inline list passed by value.
constexpr int kMaxInline = 16;
struct ExpertSrc {
    const DevExpert *table;  // device, [n_experts]  (used when ids != nullptr)
    const int32_t *ids;      // device, [k] (or [T*k] with an offset)
    DevExpert inl[kMaxInline];
};

K3_DEV DevExpert fetch_expert(const ExpertSrc &src, int j)
{
    if (src.ids) return src.table[src.ids[j]];
    return src.inl[j];
}

// 2^(e-127) for an E8M0 byte; 0 for the NaN byte 255 (the group is dropped).
K3_DEV float e8m0_scale(uint32_t e)
{
    uint32_t bits = (e == 0u) ? 0x00400000u : (e << 23);
    return (e == 255u) ? 0.0f : __uint_as_float(bits);
}

// One byte of two codes -> (even weight, odd weight) in fp32.
K3_DEV float2 e2m1x2_to_float2(uint32_t byte_in_low8)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h2)
        : "r"(byte_in_low8));
    return __half22float2(*reinterpret_cast<const __half2 *>(&h2));
}

// Four bytes (eight codes) -> four f16x2 pairs.
K3_DEV void e2m1x8_to_half2x4(uint32_t w, uint32_t &h0, uint32_t &h1, uint32_t &h2, uint32_t &h3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

K3_DEV float2 h2f2(uint32_t h)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// acc += decoded(word) . x[0..7]  (eight weights, x as four float2).
K3_DEV float2 dot8(uint32_t w, const float2 *x, float2 acc)
{
    uint32_t h0, h1, h2, h3;
    e2m1x8_to_half2x4(w, h0, h1, h2, h3);
    acc = __ffma2_rn(h2f2(h0), x[0], acc);
    acc = __ffma2_rn(h2f2(h1), x[1], acc);
    acc = __ffma2_rn(h2f2(h2), x[2], acc);
    acc = __ffma2_rn(h2f2(h3), x[3], acc);
    return acc;
}

// Dot product of one 32-group (16 bytes) with x[0..31] (16 float2), fp32.
K3_DEV float dot32(uint4 q, const float2 *x)
{
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
    a = dot8(q.x, x + 0, a);
    b = dot8(q.y, x + 4, b);
    a = dot8(q.z, x + 8, a);
    b = dot8(q.w, x + 12, b);
    return (a.x + a.y) + (b.x + b.y);
}

// Dot product of a half group (8 bytes, 16 weights) with x[0..15].
K3_DEV float dot16(uint2 q, const float2 *x)
{
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
    a = dot8(q.x, x + 0, a);
    b = dot8(q.y, x + 4, b);
    return (a.x + a.y) + (b.x + b.y);
}

// ---------------------------------------------------------------------------
// Split-activation decode (the hot path).  16 activations of one lane are
// kept as f16 halves: x * 2^s = hi + lo with hi = f16(x * 2^s) and
// lo = f16(x * 2^s - hi), 2^s chosen per 16 activations so that the largest
// is in [2^9, 2^10) (all hi, lo normal in f16).  A weight decoded by
// cvt.rn.f16x2.e2m1x2 is exact in f16, so both w * hi and w * lo are formed
// exactly and accumulated in fp32 by the mixed-precision fma.rn.f32.f16, which
// issues on the FMA pipe at full rate.  x is represented to ~2^-22 of its
// group maximum, so the products match an fp32 dot product to within fp32
// accumulation rounding.  Cost: 0.5 (decode) + 2 (FMA) instructions per
// weight, all on the ALU/FMA pipes; converting decoded weights to fp32 goes
// through the much slower f16 pipe instead.
struct XHalf16 {
    uint16_t hi[16];  // f16 bits of x * 2^s
    uint16_t lo[16];
    float inv;        // 2^-s
};

K3_DEV void split16(const float *v, XHalf16 &o)
{
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i++) m = fmaxf(m, fabsf(v[i]));
    int s = 0;
    if (m > 0.f && m < 3.0e38f) {
        int ex = ((__float_as_uint(m) >> 23) & 0xff) - 127;  // floor(log2 m) for normal m
        if (ex < -126) ex = -126;
        s = 9 - ex;
        if (s > 120) s = 120;
        if (s < -120) s = -120;
    }
    const float sc = ldexpf(1.0f, s);
    o.inv = ldexpf(1.0f, -s);
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const float a = v[i] * sc;
        const __half ha = __float2half_rn(a);
        const __half la = __float2half_rn(a - __half2float(ha));
        o.hi[i] = __half_as_ushort(ha);
        o.lo[i] = __half_as_ushort(la);
    }
}

// acc += w * x with w, x f16 (exact product), fp32 accumulate.
K3_DEV float mfma(uint16_t w, uint16_t x, float acc)
{
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(w), "h"(x));
    return acc;
}
K3_DEV uint16_t lo16(uint32_t v) { return (uint16_t)(v & 0xffffu); }
K3_DEV uint16_t hi16(uint32_t v) { return (uint16_t)(v >> 16); }

// Dot product of 16 weights (two 32-bit words of codes, low nibble first)
// with a split slice, returned in units of 2^s (multiply by x.inv).
K3_DEV float dot16_split(uint32_t w0, uint32_t w1, const XHalf16 &x)
{
    uint32_t h[8];
    e2m1x8_to_half2x4(w0, h[0], h[1], h[2], h[3]);
    e2m1x8_to_half2x4(w1, h[4], h[5], h[6], h[7]);
    float a = 0.f, b = 0.f, c = 0.f, d = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p++) {
        a = mfma(lo16(h[p]), x.hi[2 * p], a);
        b = mfma(hi16(h[p]), x.hi[2 * p + 1], b);
        c = mfma(lo16(h[p]), x.lo[2 * p], c);
        d = mfma(hi16(h[p]), x.lo[2 * p + 1], d);
    }
    return (a + b) + (c + d);
}

// Same product with only the f16-rounded activations (x.hi): one FMA per
// weight.  Activations carry 11 significant bits (relative rounding <= 2^-11),
// products and sums stay exact-product / fp32-accumulate.
K3_DEV float dot16_hi(uint32_t w0, uint32_t w1, const XHalf16 &x)
{
    uint32_t h[8];
    e2m1x8_to_half2x4(w0, h[0], h[1], h[2], h[3]);
    e2m1x8_to_half2x4(w1, h[4], h[5], h[6], h[7]);
    float a = 0.f, b = 0.f, c = 0.f, d = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p += 2) {
        a = mfma(lo16(h[p]), x.hi[2 * p], a);
        b = mfma(hi16(h[p]), x.hi[2 * p + 1], b);
        c = mfma(lo16(h[p + 1]), x.hi[2 * p + 2], c);
        d = mfma(hi16(h[p + 1]), x.hi[2 * p + 3], d);
    }
    return (a + b) + (c + d);
}
template <bool ACT16>
K3_DEV float dot16_any(uint32_t w0, uint32_t w1, const XHalf16 &x)
{
    return ACT16 ? dot16_hi(w0, w1, x) : dot16_split(w0, w1, x);
}

// Streaming loads: weights are read exactly once, keep them out of L1.
K3_DEV uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
K3_DEV uint2 ld_stream8(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}
K3_DEV uint32_t ld_stream_u8(const uint8_t *p)
{
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return (uint32_t)v;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA engine, non-tensor form) helpers.  Every wait is
// bounded by a global-timer deadline; a wait that runs out records
// K3MOE_ETIMEOUT in the device error word and returns false.
K3_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

K3_DEV void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
K3_DEV void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}
K3_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
K3_DEV uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legal wait
// try_wait with a suspend-time hint: a warp whose barrier phase has not
// completed is parked by the hardware (up to the hint) instead of spinning,
// so waiting warps do not take issue slots from working ones.
K3_DEV uint32_t mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity), "r"(20000u)
                 : "memory");
    return ok;
}
// Non-blocking: has the phase of `parity` completed?
K3_DEV bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// The waiting loop of mbar_wait, out of line: a phase that has not completed
// at the first try is waited for here, so that each of the many call sites
// inlines one try_wait (smaller kernels, fewer instruction-cache misses).
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int *err);
K3_DEV bool mbar_wait(uint32_t bar, uint32_t parity, int *err)
{
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err);
}
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, int *err)
{
    const uint64_t t0 = global_ns();
    for (uint32_t n = 1;; n++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) {
            set_device_error(err, K3MOE_ETIMEOUT);
            return false;
        }
    }
}
// Bulk copy global -> shared (16-byte aligned addresses, size a multiple of
// 16), completion counted on `bar`.
K3_DEV void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
K3_DEV uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
K3_DEV uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
K3_DEV uint32_t lds_u8(uint32_t a)
{
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
    return (uint32_t)v;
}

// Reduce N values across the 32 lanes of a warp ("transpose reduce"): after
// the call, lane l holds in v[0] the full sum of value index (l >> (5 -
// log2 N)) ... see sel_of().  N must be a power of two <= 32.
template <int N>
K3_DEV void warp_transpose_reduce(float (&v)[N], int lane)
{
    int n = N;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            const bool upper = (lane & off) != 0;
            const int h = n / 2;
#pragma unroll
            for (int i = 0; i < N / 2; i++) {
                if (i < h) {
                    float send = upper ? v[i] : v[i + h];
                    float keep = upper ? v[i + h] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n = h;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
}
// Value index whose total lane `lane` holds after warp_transpose_reduce<N>.
template <int N>
K3_DEV int sel_of(int lane)
{
    int idx = 0, n = N;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (n > 1) {
            if (lane & off) idx += n / 2;
            n /= 2;
        }
    }
    return idx;
}

// 8 x 8 transpose of 4-bit values within groups of 8 lanes: before, lane r
// of a group holds A[r][c] in nibble c; after, it holds A[c][r] in nibble c.
K3_DEV uint32_t nib_transpose8(uint32_t w, int lane)
{
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        const uint32_t M = m == 1 ? 0x0F0F0F0Fu : (m == 2 ? 0x00FF00FFu : 0x0000FFFFu);
        const int sh = 4 * m;
        const bool upper = (lane & m) != 0;
        const uint32_t send = upper ? (w & M) : ((w >> sh) & M);
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, m);
        w = upper ? ((w & (M << sh)) | recv) : ((w & M) | (recv << sh));
    }
    return w;
}

K3_DEV float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// silu(z) = z / (1 + e^-z).  The exponent is clamped at 80 so that the
// divisor stays finite (for z < -80, silu(z) is below 1e-33 in magnitude,
// negligible next to any other output of an expert): an infinite divisor
// sends the IEEE division down its slow path, which cost the epilogues half
// their time on gate values in the hundreds.  __expf and __fdividef keep the
// relative error near 1e-6, far inside every tolerance of the library.
K3_DEV float silu(float z) { return __fdividef(z, 1.0f + __expf(fminf(-z, 80.0f))); }

// Ticket of a "last CTA finishes the work" pattern: called by one thread
// after a __syncthreads that follows the CTA's global writes.  The acq_rel
// atomic publishes those writes at GPU scope (cumulatively, through the
// barrier) and, for the last CTA, makes every other CTA's writes visible;
// a fence.sc by every thread (a __threadfence) is much slower.
K3_DEV unsigned ticket_arrive(unsigned *ticket)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(ticket) : "memory");
    return old;
}

// Eight consecutive activations as fp32 (fp32 or bf16 input) and their dot
// product with eight bf16 weights (fp32 accumulation), for the router.
template <typename XT>
K3_DEV void load_x8(const XT *x, int i, float (&xv)[8]);
template <>
K3_DEV void load_x8<float>(const float *x, int i, float (&xv)[8])
{
    float4 a = __ldg(reinterpret_cast<const float4 *>(x + i));
    float4 b = __ldg(reinterpret_cast<const float4 *>(x + i + 4));
    xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
    xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
}
template <>
K3_DEV void load_x8<__nv_bfloat16>(const __nv_bfloat16 *x, int i, float (&xv)[8])
{
    uint4 a = __ldg(reinterpret_cast<const uint4 *>(x + i));
    uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        xv[2 * q] = __uint_as_float(w[q] << 16);
        xv[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
}

K3_DEV float bf16x8_dot(uint4 wv, const float (&xv)[8], float acc)
{
    uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        acc = fmaf(__uint_as_float(w[q] << 16), xv[2 * q], acc);
        acc = fmaf(__uint_as_float(w[q] & 0xffff0000u), xv[2 * q + 1], acc);
    }
    return acc;
}


// Order-preserving map of an fp32 score to uint32 (larger score -> larger key).
K3_DEV uint32_t okey(float v)
{
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The router's rule ("Running Kimi K3 locally", "How is the C engine actually
// built?", invariant 3: the bias steers the selection only, the combine
// weights come from the unbiased scores):
//  K3_ROUTER_SOFTMAX       select on logit + bias; weights = softmax of the
//                          chosen experts' logits
//  K3_ROUTER_SIGMOID       score = 1 / (1 + e^-logit); select on score + bias;
//                          weights = the chosen experts' scores
//  K3_ROUTER_SIGMOID_NORM  as K3_ROUTER_SIGMOID, weights divided by their sum
enum : int { K3_ROUTER_SOFTMAX = 0, K3_ROUTER_SIGMOID = 1, K3_ROUTER_SIGMOID_NORM = 2 };
struct Router {
    const float *bias;  // [E] selection bias, or null
    int mode;           // K3_ROUTER_*
};
K3_DEV float router_sigmoid(float l) { return 1.f / (1.f + expf(-l)); }
// selection key of expert e with logit l
K3_DEV float router_select(const Router &r, float l, int e)
{
    const float s = r.mode == K3_ROUTER_SOFTMAX ? l : router_sigmoid(l);
    return r.bias ? s + __ldg(r.bias + e) : s;
}
// combine weight of the chosen expert held by this lane (on = lane < k, l its
// logit); every lane of the warp calls it
K3_DEV float router_weight(int mode, float l, bool on)
{
    if (mode == K3_ROUTER_SOFTMAX) {
        float mx = on ? l : -INFINITY;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float ex = on ? expf(l - mx) : 0.f;
        return ex / warp_sum(ex);
    }
    const float sg = on ? router_sigmoid(l) : 0.f;
    return mode == K3_ROUTER_SIGMOID ? sg : sg / warp_sum(sg);
}

// 256 threads (threadIdx.x 0..255, synchronised by sync()) select the top k (k <= 32) of E <= 1024
// selection keys router_select(rt, logit[e], e), ties to the lower id, with the
// same result as warp_topk below: the k-th largest key is found one byte at a
// time (4 rounds of a 256-bin shared-memory histogram over the keys that
// match the prefix so far, warp-aggregated atomics, and a descending scan by
// one warp), then every key above it and the lowest-id ties at it are
// compacted in id order.  ids_out[0..k) / w_out as in warp_topk.
struct CtaTopkSmem {
    unsigned hist[256];
    unsigned cnt[2][4][8];  // per (pass, m, warp) selection counts
    int ids[32];
    unsigned prefix, need;
};
template <typename Sync, typename Logit>
K3_DEV void cta_topk_by(Logit logit_of, const Router &rt, int E, int k, int32_t *ids_out, float *w_out,
                        CtaTopkSmem &sm, Sync sync)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    uint32_t key[4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
        const int e = t + 256 * m;
        key[m] = 0u;  // below every real key
        if (e < E) key[m] = okey(router_select(rt, logit_of(e), e));
    }
    uint32_t prefix = 0u, mask = 0u;
    unsigned need = (unsigned)k;
#pragma unroll 1
    for (int r = 0; r < 4; r++) {
        const int shift = 24 - 8 * r;
        sm.hist[t] = 0u;
        sync();
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const bool in = (t + 256 * m < E) && (key[m] & mask) == prefix;
            const unsigned act = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned dg = (key[m] >> shift) & 255u;
                const unsigned peers = __match_any_sync(act, dg);
                if (lane == __ffs(peers) - 1) atomicAdd(&sm.hist[dg], (unsigned)__popc(peers));
            }
        }
        sync();
        if (warp == 0) {
            // lane l owns bins 255-8l .. 248-8l (descending)
            unsigned hb[8], own = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                hb[i] = sm.hist[255 - 8 * lane - i];
                own += hb[i];
            }
            unsigned incl = own;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            const unsigned excl = incl - own;
            if (excl < need && incl >= need) {
                unsigned cum = excl;
                for (int i = 0; i < 8; i++) {
                    if (cum + hb[i] >= need) {
                        sm.prefix = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
                        sm.need = need - cum;
                        break;
                    }
                    cum += hb[i];
                }
            }
        }
        sync();
        prefix = sm.prefix;
        need = sm.need;
        mask |= 255u << shift;
    }
    // prefix = the k-th largest key; take the `need` lowest-id ties at it
    const uint32_t T = prefix;
    const unsigned lt = (1u << lane) - 1u;
    unsigned eqb[4], rank_eq[4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
        eqb[m] = __ballot_sync(0xffffffffu, (t + 256 * m < E) && key[m] == T);
        if (lane == 0) sm.cnt[0][m][warp] = __popc(eqb[m]);
    }
    sync();
    if (warp == 0) {  // exclusive prefix over (m, warp) = id order
        const unsigned c = sm.cnt[0][lane >> 3][lane & 7];
        unsigned incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        sm.cnt[0][lane >> 3][lane & 7] = incl - c;
    }
    sync();
    unsigned selb[4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
        rank_eq[m] = sm.cnt[0][m][warp] + __popc(eqb[m] & lt);
        const bool sel = (t + 256 * m < E) &&
                         (key[m] > T || (((eqb[m] >> lane) & 1u) && rank_eq[m] < need));
        selb[m] = __ballot_sync(0xffffffffu, sel);
        if (lane == 0) sm.cnt[1][m][warp] = __popc(selb[m]);
    }
    sync();
    if (warp == 0) {
        const unsigned c = sm.cnt[1][lane >> 3][lane & 7];
        unsigned incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        sm.cnt[1][lane >> 3][lane & 7] = incl - c;
    }
    sync();
#pragma unroll
    for (int m = 0; m < 4; m++)
        if ((selb[m] >> lane) & 1u) sm.ids[sm.cnt[1][m][warp] + __popc(selb[m] & lt)] = t + 256 * m;
    sync();
    if (warp == 0) {
        const int my_id = (lane < k) ? sm.ids[lane] : 0;
        const float wv = router_weight(rt.mode, (lane < k) ? logit_of(my_id) : 0.f, lane < k);
        if (lane < k) {
            ids_out[lane] = my_id;
            w_out[lane] = wv;
        }
    }
}
// A CTA of at least eight warps selects the top k (k <= 16) of E <= 1024
// selection keys okey(router_select(rt, logit_of(e), e)), ties to the lower
// id, with the same result as cta_topk_by and warp_topk; ids_out[0..k)
// receives the ids in ascending order (the combine weights are left to the
// caller, see router_weight).  Words key << 32 | (2^32 - 1 - id) order
// exactly like (key descending, id ascending).  Warp w < 8 holds the
// m = ceil(E / 8) ids [w m, w m + m), lane l the ids w m + l + 32 r (r < 4:
// consecutive lanes read consecutive logits).
//  1. T_w = the R-th largest (R = ceil(k / 8)) of warp w's lane maxima, the
//     lanes tied at a maximum dropping out together, so that at least R of
//     the warp's keys are >= T_w; T = the smallest T_w.  At least 8 R >= k
//     keys are >= T, so the k largest words all have keys >= T.
//  2. The words whose keys are >= T (a few dozen for untied keys) go to
//     shared memory, and each one's place is the number of those words
//     larger than it (eight lanes a word, each comparing it with every eighth
//     word): the k whose place is below k are the result.
//  3. If more than 128 keys are >= T (many ties at T, or fewer than R keys in
//     some warp), each warp takes its k largest words instead (k rounds of an
//     exact warp maximum) and the 8 k candidates are ranked the same way.
// Then warp 0 puts the k ids in ascending order.  Every thread of the CTA
// calls it; sync() is a barrier over all of them.
struct CtaTopkRedSmem {
    alignas(16) uint64_t cand[128];  // candidate words (0: unused)
    alignas(16) uint32_t thr[8];     // T_w
    int32_t ids[16];                 // the k winners by place
    int32_t cnt;                     // candidates
};
K3_DEV uint64_t topk_word(uint32_t key, int id, int E)
{
    return id < E ? ((uint64_t)key << 32) | (uint64_t)(0xffffffffu - (uint32_t)id) : 0ull;
}
K3_DEV int topk_word_id(uint64_t w) { return (int)(0xffffffffu - (uint32_t)w); }
K3_DEV void topk_sort2(uint64_t &a, uint64_t &b)
{
    const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}
// the warp's largest of the lanes' words w (exact: key, then the lower id)
K3_DEV uint64_t warp_max_word(uint64_t w)
{
    const uint32_t hk = (uint32_t)(w >> 32), lk = (uint32_t)w;
    const uint32_t mk = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t ml = __reduce_max_sync(0xffffffffu, hk == mk ? lk : 0u);
    return ((uint64_t)mk << 32) | ml;
}
template <typename Sync, typename Logit>
K3_DEV void cta_topk_red(Logit logit_of, const Router &rt, int E, int k, int32_t *ids_out, CtaTopkRedSmem &sm,
                         Sync sync)
{
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int R = (k + 7) >> 3, m = (E + 7) >> 3;
    const unsigned lt = (1u << lane) - 1u;
    uint32_t key[4];
    unsigned valid = 0u;  // bit r: slot r holds an expert
    if (t < 128) sm.cand[t] = 0ull;
    if (warp < 8) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int j = lane + 32 * r, e = warp * m + j;
            key[r] = 0u;
            if (j < m && e < E) {
                key[r] = okey(router_select(rt, logit_of(e), e));
                valid |= 1u << r;
            }
        }
        uint32_t lk = 0u;
#pragma unroll
        for (int r = 0; r < 4; r++)
            if ((valid >> r) & 1u) lk = max(lk, key[r]);
        uint32_t tw = 0u;
        for (int i = 0; i < R; i++) {
            tw = __reduce_max_sync(0xffffffffu, lk);
            if (lk == tw) lk = 0u;
        }
        if (lane == 0) sm.thr[warp] = tw;
        if (t == 0) sm.cnt = 0;
    }
    sync();
    if (warp < 8) {
        const uint4 ta = *reinterpret_cast<const uint4 *>(&sm.thr[0]);
        const uint4 tb = *reinterpret_cast<const uint4 *>(&sm.thr[4]);
        const uint32_t T = min(min(min(ta.x, ta.y), min(ta.z, ta.w)), min(min(tb.x, tb.y), min(tb.z, tb.w)));
        unsigned b[4];
        int c = 0;
#pragma unroll
        for (int r = 0; r < 4; r++) {
            b[r] = __ballot_sync(0xffffffffu, ((valid >> r) & 1u) && key[r] >= T);
            c += __popc(b[r]);
        }
        int base = 0;
        if (lane == 0 && c) base = atomicAdd(&sm.cnt, c);
        base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
        for (int r = 0; r < 4; r++) {
            if ((b[r] >> lane) & 1u) {
                const int pos = base + __popc(b[r] & lt);
                if (pos < 128) sm.cand[pos] = topk_word(key[r], warp * m + lane + 32 * r, E);
            }
            base += __popc(b[r]);
        }
    }
    sync();
    int n = sm.cnt;
    if (n > 128) {
        sync();  // every thread has read the count
        if (warp < 8) {
            uint64_t w[4];
#pragma unroll
            for (int r = 0; r < 4; r++)
                w[r] = ((valid >> r) & 1u) ? topk_word(key[r], warp * m + lane + 32 * r, E) : 0ull;
            topk_sort2(w[0], w[1]);
            topk_sort2(w[2], w[3]);
            topk_sort2(w[0], w[2]);
            topk_sort2(w[1], w[3]);
            topk_sort2(w[1], w[2]);
            uint64_t mine = 0ull;
            for (int i = 0; i < k; i++) {
                const uint64_t M = warp_max_word(w[0]);
                if (lane == i) mine = M;
                if (w[0] == M) {  // the lane holding it moves on to its next
                    w[0] = w[1];
                    w[1] = w[2];
                    w[2] = w[3];
                    w[3] = 0ull;
                }
            }
            if (lane < 16) sm.cand[16 * warp + lane] = mine;
        }
        n = 128;
        sync();
    }
    {
        const int s = lane & 7, n8 = (n + 7) >> 3, per = (int)(blockDim.x >> 5) * 4;
        for (int c0 = 0; c0 < n; c0 += per) {
            const int c = c0 + warp * 4 + (lane >> 3);
            const uint64_t vc = c < n ? sm.cand[c] : 0ull;
            int a = 0;
            for (int q = 0; q < n8; q++) a += (int)(sm.cand[8 * q + s] > vc);
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            if (s == 0 && vc != 0ull && a < k) sm.ids[a] = topk_word_id(vc);
        }
    }
    sync();
    if (warp == 0) {
        // each winner's place in ascending id order
        const int rid = lane < k ? sm.ids[lane] : 0x7fffffff;
        int rank = 0;
#pragma unroll
        for (int q = 0; q < 16; q++) rank += (int)(__shfl_sync(0xffffffffu, rid, q) < rid);
        if (lane < k) ids_out[rank] = rid;
    }
}

// logits in global memory (ld.cg: other CTAs may have written them)
template <typename Sync>
K3_DEV void cta_topk(const float *logit, const Router &rt, int E, int k, int32_t *ids_out, float *w_out,
                     CtaTopkSmem &sm, Sync sync)
{
    cta_topk_by([&](int e) { return __ldcg(logit + e); }, rt, E, k, ids_out, w_out, sm, sync);
}

// One warp selects the top k (k <= 32) of E <= 1024 selection keys
// router_select(rt, logit[e], e), ties to the lower id: a radix search for
// the k-th largest key (32 rounds of one count and one warp reduction), then
// every key above it and the lowest-id ties at it.  ids_out[0..k) receives
// the ids in ascending order and w_out the router's weights from the
// UNBIASED scores ("Running Kimi K3 locally", invariant 3).  logit is read
// with ld.cg (other CTAs may have written it); ids_out is read back by the
// warp.
K3_DEV void warp_topk(const float *logit, const Router &rt, int E, int k, int32_t *ids_out,
                      float *w_out, int lane)
{
    uint32_t key[32];
#pragma unroll
    for (int q = 0; q < 32; q++) {
        const int e = lane + 32 * q;
        key[q] = 0u;  // below every real key (okey(-inf) = 0x007fffff)
        if (e < E) key[q] = okey(router_select(rt, __ldcg(logit + e), e));
    }
    uint32_t T = 0u;  // largest T with count(key >= T) >= k
    for (int b = 31; b >= 0; b--) {
        const uint32_t cand = T | (1u << b);
        uint32_t c0 = 0, c1 = 0;
#pragma unroll
        for (int q = 0; q < 32; q += 2) {
            c0 += key[q] >= cand;
            c1 += key[q + 1] >= cand;
        }
        if (__reduce_add_sync(0xffffffffu, c0 + c1) >= (unsigned)k) T = cand;
    }
    uint32_t cgt = 0;
#pragma unroll
    for (int q = 0; q < 32; q++) cgt += key[q] > T;
    const int need = k - (int)__reduce_add_sync(0xffffffffu, cgt);
    const uint32_t lt = (1u << lane) - 1u;
    int eq_before = 0, sel_before = 0;
#pragma unroll
    for (int q = 0; q < 32; q++) {
        const int e = lane + 32 * q;
        const bool eq = (e < E) && key[q] == T;
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        const bool pick_eq = eq && (eq_before + __popc(beq & lt)) < need;
        const bool sel = ((e < E) && key[q] > T) || pick_eq;
        const unsigned bsel = __ballot_sync(0xffffffffu, sel);
        if (sel) ids_out[sel_before + __popc(bsel & lt)] = e;
        eq_before += __popc(beq);
        sel_before += __popc(bsel);
    }
    __syncwarp();
    const int my_id = (lane < k) ? ids_out[lane] : 0;
    const float wv = router_weight(rt.mode, (lane < k) ? __ldcg(logit + my_id) : 0.f, lane < k);
    if (lane < k) w_out[lane] = wv;
    __syncwarp();
}


}  // namespace k3
