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

// Spread eight 2-bit digits (digit q at bits 2q + 1 .. 2q of x) into the
// low two bits of eight nibbles (digit q to nibble q).
K3_DEV uint32_t spread_digits(uint32_t x)
{
    x &= 0xFFFFu;
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    x = (x | (x << 2)) & 0x33333333u;
    return x;
}

// One warp encodes one 32-block of v (lane i holds element i) as MX_N E2M1
// pieces into img / sf.  With E the biased exponent of the block's largest
// magnitude (at least 1), every |v| becomes the 32-bit integer
// M = |v| * 2^(158 - E) (exact for |v| >= 2^(E - 135), rounded to the
// nearest integer below that, so the error is at most 2^(E - 159): 2^-32 of
// the block's scale), and piece p is the p-th base-4 digit of M from the top,
// d_p = (M >> (30 - 2p)) & 3, an E2M1 magnitude d_p / 2 (codes 0-3) with the
// scale 2^(E - 127 - 2p) (E8M0 byte E - 2p; pieces whose byte would be
// negative are left out, all their digits standing for less than 2^-126).
// The sign goes into every nibble (a zero digit becomes -0).  So
// sum_p piece_p = sign * M * 2^(E - 158), and piece 0 carries the largest
// part, as the epilogues' order of summation expects.  A block holding a
// non-finite value gets scale byte 255 (NaN) in every piece, so the products
// carry the NaN on; an all-zero block gets codes 0.  No step depends on the
// previous piece: one block maximum, then bit arithmetic per lane, an 8 x 8
// nibble transpose within each group of eight lanes (lane j of group g: word
// g of pieces j and 8 + j), two word stores per lane and one scale byte per
// piece.
K3_DEV void mx_encode_block(float v, int lane, int b, uint8_t *img, uint8_t *sf)
{
    const uint32_t bits = __float_as_uint(v), ab = bits & 0x7fffffffu;
    const bool bad = __any_sync(0xffffffffu, ab >= 0x7f800000u);
    const uint32_t mb = __reduce_max_sync(0xffffffffu, ab);
    const int E = max((int)(mb >> 23), 1);
    uint32_t c0 = 0u, c1 = 0u, sbyte = 127u;
    if (bad) {
        sbyte = 255u;
    } else if (mb != 0u) {
        const int ev = max((int)(ab >> 23), 1);
        const uint32_t m24 = (ab & 0x7fffffu) | ((ab >> 23) ? 0x800000u : 0u);
        const int sh = ev - E + 8;  // <= 8
        uint32_t M;
        if (sh >= 0) M = m24 << sh;
        else M = -sh < 32 ? (m24 + (1u << (-sh - 1))) >> -sh : 0u;
        // digit p of M (from the top) to nibble p: reverse the digit order
        // (bit reversal, then swap the two bits of each digit), then spread
        uint32_t R = __brev(M);
        R = ((R >> 1) & 0x55555555u) | ((R & 0x55555555u) << 1);
        c0 = spread_digits(R);        // digits 0-7
        c1 = spread_digits(R >> 16);  // digits 8-15
        if (E < 2 * (MX_N - 1)) {     // pieces whose scale byte E - 2p would be negative
            const int pmax = E >> 1;  // last piece with E - 2p >= 0
            const uint64_t keep = pmax >= 15 ? ~0ull : ((1ull << (4 * (pmax + 1))) - 1ull);
            c0 &= (uint32_t)keep;
            c1 &= (uint32_t)(keep >> 32);
        }
        if (bits >> 31) {
            c0 |= 0x88888888u;
            c1 |= 0x88888888u;
        }
        sbyte = (uint32_t)max(E - 2 * lane, 0);
    }
    const int j = lane & 7, g = lane >> 3;
    const uint32_t w0 = nib_transpose8(c0, lane), w1 = nib_transpose8(c1, lane);
    *(uint32_t *)(img + mx_img_off(j, b, g)) = w0;
    *(uint32_t *)(img + mx_img_off(8 + j, b, g)) = w1;
    if (lane < MX_N) sf[mx_sf_off(lane, b)] = (uint8_t)sbyte;
}

}  // namespace k3
