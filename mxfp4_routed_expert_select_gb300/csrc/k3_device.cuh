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

K3_DEV float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

K3_DEV float silu(float z) { return z / (1.0f + expf(-z)); }

// Device error word (bounded waits that ran out write K3MOE_ETIMEOUT here);
// one int per device, allocated by the host side (k3::device_error_word()).
K3_DEV void set_device_error(int *err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

}  // namespace k3
