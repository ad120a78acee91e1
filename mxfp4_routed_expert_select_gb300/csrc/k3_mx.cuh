// k3_mx.cuh -- E2M1 pieces of an fp32 vector, the B operand of the
// block-scaled (kind::mxf4) tensor-core products (see k3_mx.cu).
#pragma once
#include "k3_device.cuh"

namespace k3 {

constexpr int MX_N = 16;  // pieces = B rows = MMA N

// byte offset of (piece p, 32-block b, word w) in a B image and of the scale
// byte of (p, b) in a scale-atom image
K3_DEV size_t mx_img_off(int p, int b, int w)
{
    return (size_t)(b >> 3) * (MX_N * 128) + p * 128 + ((((b & 7) ^ (p & 7))) << 4) + 4 * w;
}
K3_DEV size_t mx_sf_off(int p, int b) { return (size_t)(b >> 2) * 512 + 16 * p + (b & 3); }

// One warp encodes one 32-block of v (lane i holds element i) as MX_N E2M1
// pieces into img / sf.  A block holding a non-finite value gets scale byte
// 255 (NaN) in every piece, so the products carry the NaN on.
K3_DEV void mx_encode_block(float r, int lane, int b, uint8_t *img, uint8_t *sf)
{
    const bool bad = __any_sync(0xffffffffu, !(fabsf(r) <= 3.4028235e38f));
#pragma unroll 1
    for (int p = 0; p < MX_N; p++) {
        // block maximum of |r|: non-negative floats order like their bits
        const uint32_t mb = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(r)));
        const float m = __uint_as_float(mb);
        uint32_t sbyte = 127u, code = 0u;
        if (bad) {
            sbyte = 255u;
        } else if (m > 0.f) {
            const int ex = (int)max(mb >> 23, 1u) - 126;  // 2^(ex-1) <= m < 2^ex (m normal)
            int s = (m <= 0.75f * __int_as_float((127 + min(ex, 127)) << 23)) ? ex - 3 : ex - 2;
            s = min(max(s, -126), 126);
            sbyte = (uint32_t)(s + 127);
            const float a = fabsf(r) * __int_as_float((127 - s) << 23);  // |r| / 2^s, exact
            code = (a >= 0.25f) + (a >= 0.75f) + (a >= 1.25f) + (a >= 1.75f) + (a >= 2.5f) + (a >= 3.5f) +
                   (a >= 5.0f);
            const float qv = code < 4u ? 0.5f * (float)code : (code == 7u ? 6.f : (float)code - 2.f);
            const float q = copysignf(qv, r) * __int_as_float((127 + s) << 23);
            if (r < 0.f && code) code |= 8u;
            r -= q;  // exact: q is r rounded on a grid no finer than r's own
        }
        uint32_t word = code << (4 * (lane & 7));
        word |= __shfl_xor_sync(0xffffffffu, word, 1);
        word |= __shfl_xor_sync(0xffffffffu, word, 2);
        word |= __shfl_xor_sync(0xffffffffu, word, 4);
        if ((lane & 7) == 0) *(uint32_t *)(img + mx_img_off(p, b, lane >> 3)) = word;
        if (lane == 0) sf[mx_sf_off(p, b)] = (uint8_t)sbyte;
    }
}

}  // namespace k3
