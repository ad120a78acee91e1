// k3_tc.cu -- grouped expert products on the tensor cores (tcgen05 + TMEM).
//
// Multi-token batches (decode batches, prefill) group the (token, slot) pairs
// by expert, so every expert matrix meets a block of tokens and the work is a
// dense grouped contraction.  The pages give the per-expert products
// ("kimi-k3-in-c" explainer, "Reduction one": E2M1 codes, one E8M0 scale per
// 32 weights); here they run as MMAs:
//
//   weights  E2M1 * 2^(e-127) is exact in bf16 (2 significant bits, bf16 has
//            8 exponent bits), so decode warps turn the packed nibbles into
//            bf16 in shared memory, exactly, in the 128-byte-swizzled K-major
//            layout the MMA reads.  The packed bytes never exist as floats in
//            global memory.
//   tokens   fp32 activations are split x = hi + lo, hi = bf16(x),
//            lo = bf16(x - hi) (16 significant bits, relative 2^-17); both
//            halves are columns of the same MMA and are added in the
//            epilogue.  bf16 activations need no split.
//   h        the SwiGLU output is split the same way for the down product.
//   products bf16 x bf16 -> fp32 accumulation in TMEM (tcgen05.mma
//            kind::f16, M = 128 weight rows, N = the tile's token columns).
//
// Per step: k3_tc_plan cuts every expert's pairs into tiles of at most TN
// tokens; k3_tc_gather writes each tile's token rows (bf16, pre-swizzled,
// k-step-major so a k-step of a tile is one contiguous block); k3_tc_expert<0>
// computes h for (tile, 128 rows of f) units; k3_tc_expert<1> computes the
// down product for (tile, 128 rows of d) units and adds w * y into the output
// (fp32 atomics: the order of the k additions of a token is not fixed).
//
// One persistent CTA per SM, 15 warps:
//   warp 0      TMA of packed weight tiles (128 rows x 128 bytes per matrix,
//               one tensor map per expert matrix) into a staging ring
//   warp 1      bulk copies of token tiles, one per k-step, into a ring of
//               2 KB slots (a k-step takes N/16 slots, so narrow tiles run
//               up to 16 k-steps ahead and wide ones as far as space allows)
//   warp 2      TMEM owner; lane 0 issues the MMAs and commits
//   warps 3-10  decoders: staged nibbles -> bf16, two threads per weight row
//   warps 11-14 epilogue: TMEM -> registers -> SwiGLU / weighted combine
// Every wait is bounded (2 s); a timeout sets the device error word, the CTA
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "k3_tcgen05.cuh"

namespace k3 {

// One tile: up to TN tokens of one expert.  Token rows (nx of them, from
// xrow0; `split` pieces of P = n rounded up to 8 rows each, or one block of
// n rows rounded up to 16 when split is 1) and h rows (nh from hrow0: bf16
// hi and lo, nh = 2P, or four e4m3 pieces, nh = 4P).
struct TcTile {
    int32_t expert, pair_begin, n, nx, nh, xrow0, hrow0, split;
};

namespace {

constexpr int TC_M = 128;           // weight rows per unit (MMA M)
constexpr int TC_SS = 256;          // K per staging step: 128 packed bytes per row
constexpr int W_PK = 0, W_B = 1, W_MMA = 2, W_DEC = 3;
constexpr int TC_NB = 16;           // token k-steps in flight at most
constexpr int TC_SLOT = 2048;       // token ring granularity: 16 rows x 128 bytes
constexpr uint32_t TC_TMEM_COLS = 512;

// PH: 0 = gate/up + SwiGLU, 1 = down + combine.  KD: operand kind, 0 = bf16
// (kind::f16, a k-step is 64 of K), 1 = e4m3 (kind::f8f6f4, 128 of K).
template <int PH, int KD>
struct TcCfg {
    static constexpr int NA = PH == 0 ? 2 : 1;                // matrices per unit
    static constexpr int SA = PH == 0 ? 3 : 4;                // decoded-weight stages
    static constexpr int SP = PH == 0 ? 2 : 3;                // packed staging stages
    static constexpr int KSK = KD ? 128 : 64;                 // K per k-step (one 128-byte row)
    static constexpr int KPS = TC_SS / KSK;                   // k-steps per staging step
    static constexpr int GPK = KSK / 32;                      // 32-groups per k-step
    static constexpr int NSLOT = PH == 0 ? (KD ? 30 : 32) : (KD ? 54 : 56);  // token ring slots
    static constexpr int BMAX = PH == 0 ? 128 : 256;          // token rows per k-step
    static constexpr int A_BYTES = NA * TC_M * 128;
    static constexpr int PK_BYTES = NA * TC_M * 128;          // swizzled like the operands
    static constexpr int PK_OFF = SA * A_BYTES;
    static constexpr int B_OFF = PK_OFF + SP * PK_BYTES;
    static constexpr int LUT_OFF = B_OFF + NSLOT * TC_SLOT;   // e4m3 decode tables (KD = 1)
    static constexpr int BAR_OFF = LUT_OFF + (KD ? 256 * 8 : 0);
    static constexpr int NBARS = 2 * SP + 2 * SA + 2 * 16 + 5;  // mbarriers (see the kernel)
    static constexpr int BAR_BYTES = 768;                     // mbarriers, token ring offsets, TMEM slot, flag
    static constexpr int SMEM = BAR_OFF + BAR_BYTES + 1024;   // + alignment slack
    static_assert(NBARS * 8 + 16 * 4 + 8 <= BAR_BYTES, "barrier block");
    static constexpr int DEC = 8;                             // decoder warps
    static constexpr int IPP = NA * GPK / (DEC / 4);          // 32-groups per thread per k-step
    static constexpr int W_EPI = W_DEC + DEC;
    static constexpr int THREADS = (W_EPI + 4) * 32;
    static_assert(IPP >= 1 && GPK % IPP == 0, "decoder split");
    static_assert(BMAX / 16 <= NSLOT / 2, "token ring too small");
    static_assert(SMEM <= 232448, "shared memory");
};

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = n (multiple of 16, <= 256).
K3_DEV uint32_t bf16_idesc(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TC_M >> 4) << 24);
}
// kind::f8f6f4 with e4m3 A and B (format code 0), otherwise the same fields.
K3_DEV uint32_t e4m3_idesc(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TC_M >> 4) << 24); }
// One k-step (64 of K) of D (+)= A * B^T: four K = 16 MMAs on consecutive
// 32-byte slices of A and B, A and B given by the low halves of their
// descriptors.  Executed by the whole warp; elect.sync picks the one lane
// that issues.  The per-MMA offsets are added inside one asm block, so the
// operands that vary from one k-step to the next are moved once per block
// (an MMA whose descriptor is recomputed outside costs about 90 cycles more).
// Both kinds read 32 bytes of K per MMA (16 bf16 or 32 e4m3 values).
#define K3_MMA4(KIND, TD, AL, BL)                                                                            \
    "mov.b64 da, {" AL ", %5};\n\tmov.b64 db, {" BL ", %5};\n\t"                                          \
    "@e tcgen05.mma.cta_group::1." KIND " [" TD "], da, db, %3, p;\n\t"                                     \
    "add.u32 a, " AL ", 2;\n\tadd.u32 b, " BL ", 2;\n\tmov.b64 da, {a, %5};\n\tmov.b64 db, {b, %5};\n\t" \
    "@e tcgen05.mma.cta_group::1." KIND " [" TD "], da, db, %3, 1;\n\t"                                     \
    "add.u32 a, " AL ", 4;\n\tadd.u32 b, " BL ", 4;\n\tmov.b64 da, {a, %5};\n\tmov.b64 db, {b, %5};\n\t" \
    "@e tcgen05.mma.cta_group::1." KIND " [" TD "], da, db, %3, 1;\n\t"                                     \
    "add.u32 a, " AL ", 6;\n\tadd.u32 b, " BL ", 6;\n\tmov.b64 da, {a, %5};\n\tmov.b64 db, {b, %5};\n\t" \
    "@e tcgen05.mma.cta_group::1." KIND " [" TD "], da, db, %3, 1;\n\t"
#define K3_KSTEP1(KIND)                                                                                      \
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t.reg .b32 a, b;\n\t"                      \
                 "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t" K3_MMA4(KIND, "%0", "%1", "%2") "}" \
                 ::"r"(td), "r"(alo), "r"(blo), "r"(idesc), "r"(acc), "r"(SW128_HI)                           \
                 : "memory")
// Two matrices (gate, up) against the same B: A of the second matrix is
// 16 KB further (+1024 in the descriptor), its accumulator 128 columns on.
#define K3_KSTEP2(KIND)                                                                                      \
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t.reg .b32 a, b, a1, t1;\n\t"              \
                 "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"                                   \
                 "add.u32 a1, %1, 1024;\n\tadd.u32 t1, %0, 128;\n\t" K3_MMA4(KIND, "%0", "%1", "%2")           \
                     K3_MMA4(KIND, "t1", "a1", "%2") "}" ::"r"(td),                                           \
                 "r"(alo), "r"(blo), "r"(idesc), "r"(acc), "r"(SW128_HI)                                      \
                 : "memory")
template <int NA, int KD>
K3_DEV void mma_kstep(uint32_t td, uint32_t alo, uint32_t blo, uint32_t idesc, uint32_t acc)
{
    if constexpr (NA == 2 && KD == 0) K3_KSTEP2("kind::f16");
    if constexpr (NA == 2 && KD == 1) K3_KSTEP2("kind::f8f6f4");
    if constexpr (NA == 1 && KD == 0) K3_KSTEP1("kind::f16");
    if constexpr (NA == 1 && KD == 1) K3_KSTEP1("kind::f8f6f4");
}
#undef K3_KSTEP1
#undef K3_KSTEP2
#undef K3_MMA4
K3_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// f16 bits of 2^(e-127) when that is a normal f16 (e in [113, 142]), else 0
// with ok = false.  The NaN byte 255 gives 0 (the group is dropped), ok.
K3_DEV uint16_t e8m0_f16(uint32_t e, bool &ok)
{
    ok = true;
    if (e == 255u) return 0;
    if (e >= 113u && e <= 142u) return (uint16_t)((e - 112u) << 10);
    ok = false;
    return 0;
}

// Eight codes (one word) times the group scale -> eight exact bf16 values.
// Fast form: f16 code * f16 scale in fp32 (exact), the bf16 is the high half.
K3_DEV uint4 decode8_bf16(uint32_t w, uint16_t sc)
{
    uint32_t h0, h1, h2, h3;
    e2m1x8_to_half2x4(w, h0, h1, h2, h3);
    uint4 o;
    o.x = prmt(__float_as_uint(mfma(lo16(h0), sc, 0.f)), __float_as_uint(mfma(hi16(h0), sc, 0.f)), 0x7632u);
    o.y = prmt(__float_as_uint(mfma(lo16(h1), sc, 0.f)), __float_as_uint(mfma(hi16(h1), sc, 0.f)), 0x7632u);
    o.z = prmt(__float_as_uint(mfma(lo16(h2), sc, 0.f)), __float_as_uint(mfma(hi16(h2), sc, 0.f)), 0x7632u);
    o.w = prmt(__float_as_uint(mfma(lo16(h3), sc, 0.f)), __float_as_uint(mfma(hi16(h3), sc, 0.f)), 0x7632u);
    return o;
}
// General form for any scale byte: fp32 multiply by 2^(e-127).
K3_DEV uint4 decode8_bf16_any(uint32_t w, float s)
{
    uint32_t h[4];
    e2m1x8_to_half2x4(w, h[0], h[1], h[2], h[3]);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float2 f = h2f2(h[i]);
        o[i] = prmt(__float_as_uint(f.x * s), __float_as_uint(f.y * s), 0x7632u);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Eight codes (one word) -> eight e4m3 bytes through a per-scale table of
// the eight magnitudes (t[m] = e4m3 of E2M1 magnitude m times 2^(e-127),
// bytes 0-3 in tlo, 4-7 in thi): the magnitudes are byte lookups with the
// nibbles as selectors, and each nibble's sign (bit 3) lands on bit 7 of its
// byte by interleaving the bytes of w << 4 (even nibbles) and w (odd ones).
K3_DEV uint2 decode8_e4m3(uint32_t w, uint32_t tlo, uint32_t thi)
{
    const uint32_t mag = w & 0x77777777u;
    const uint32_t w4 = w << 4;
    uint2 o;
    o.x = prmt(tlo, thi, mag) | (prmt(w4, w, 0x5140u) & 0x80808080u);
    o.y = prmt(tlo, thi, mag >> 16) | (prmt(w4, w, 0x7362u) & 0x80808080u);
    return o;
}

// out[0..3] += v0..v3 with one vector reduction (16-byte aligned address).
K3_DEV void red_add_v4(float *out, float v0, float v1, float v2, float v3)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(v0), "f"(v1), "f"(v2), "f"(v3)
                 : "memory");
}
// Transposes an 8 x 8 block held by groups of 8 lanes: before, lane g holds
// v[i] = A[g][i]; after, v[i] = A[i][g] (three butterfly exchange stages).
K3_DEV void transpose8(float (&v)[8], int lane)
{
    const int g = lane & 7;
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; i++) {
            if ((i & m) == 0) {
                const bool upper = (g & m) != 0;
                const float send = upper ? v[i] : v[i | m];
                const float recv = __shfl_xor_sync(0xffffffffu, send, m);
                if (upper)
                    v[i] = recv;
                else
                    v[i | m] = recv;
            }
        }
    }
}

K3_DEV uint32_t bf16_rn_bits(float v) { return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// Scale of piece 0 of e4m3 pieces for values of largest magnitude m:
// 2^(x - 8) for m = mant 2^x, mant in [0.5, 1) (so |v| / scale < 256, below
// the e4m3 maximum 448); 1 for m = 0.
K3_DEV float piece_scale(float m)
{
    int ex = 0;
    frexpf(m, &ex);
    return m > 0.f ? ldexpf(1.f, ex - 8) : 1.f;
}
K3_DEV float h_scale(unsigned mbits) { return piece_scale(__uint_as_float(mbits)); }

// Rows of a tile of n tokens.  An operand split in np pieces keeps piece c
// in rows [c P, c P + n), P = n rounded up to 8 (bf16 hi/lo: np = 2; e4m3
// pieces: np = 2 or 4); every MMA width is a multiple of 16.
K3_DEV int tile_p(int n) { return (n + 7) & ~7; }
K3_DEV int tile_nx(int n, int np) { return np > 1 ? np * tile_p(n) : (n + 15) & ~15; }
K3_DEV int tile_nh(int n, int nph) { return nph * tile_p(n); }

struct TcArgs {
    const TcTile *tiles;
    const int32_t *n_tiles;
    const DevExpert *table;
    const CUtensorMap *maps;  // [E][3]: gate, up, down packed planes
    const uint8_t *Bsrc;      // token rows (phase 0) or h rows (phase 1)
    uint8_t *Hg;              // phase 0 output
    float *out;               // phase 1 output [T x d]
    const int32_t *perm;
    const float *wsel;
    const float *tscale;      // e4m3 token pieces: per-token scale of piece 0
    float *hf;                // e4m3 down: h in fp32, [pair][f] in tile order
    unsigned *hmax;           // e4m3 down: per pair, bits of max |h| (non-negative floats order as ints)
    int k, d, f;
    int *err;
};

}  // namespace

template <int PH, int KD>
__global__ void __launch_bounds__(TcCfg<PH, KD>::THREADS, 1) k3_tc_expert(const TcArgs a)
{
    using C = TcCfg<PH, KD>;
    constexpr int W_EPI = C::W_EPI;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(sm);
    uint64_t *bars = (uint64_t *)(sm + C::BAR_OFF);
    const int B_PKF = 0, B_PKE = B_PKF + C::SP, B_AF = B_PKE + C::SP, B_AE = B_AF + C::SA, B_BF = B_AE + C::SA,
              B_BE = B_BF + TC_NB, B_ACCF = B_BE + TC_NB, B_ACCE = B_ACCF + 2, B_FIN = B_ACCE + 2,
              NBARS = B_FIN + 1;
    static_assert(2 * C::SP + 2 * C::SA + 2 * TC_NB + 5 == C::NBARS, "barrier count");
    volatile uint32_t *boff = (volatile uint32_t *)(bars + NBARS);  // [TC_NB] token ring offsets
    uint32_t *tmem_slot = (uint32_t *)(boff + TC_NB);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(bars + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = PH == 0 ? a.d : a.f;     // reduction length
    const int ROWS = PH == 0 ? a.f : a.d;  // weight rows per matrix
    const int nrb = ROWS / TC_M;
    const int nss = K / TC_SS;
    const int nks = K / C::KSK;
    // Units are (tile, 128-row block) pairs, unit u = tile u / nrb, row
    // block u % nrb.  Every role walks the same units (CTA index, += number
    // of CTAs) and fetches the next unit's tile record one unit ahead; every
    // CTA copies its own token (or h) rows.
    const int ncl = (int)gridDim.x, cid = (int)blockIdx.x;
    const int gpt = nrb;                        // units per tile
    const int n_groups = *a.n_tiles * gpt;
    auto unit_of = [&](int ug) { return ug; };
    auto tile_at = [&](int ug) -> TcTile {
        TcTile t = {};
        if (ug < n_groups) t = a.tiles[ug / gpt];
        return t;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::SP; i++) {
            mbar_init(bar(B_PKF + i), 1);
            mbar_init(bar(B_PKE + i), C::DEC);
        }
        for (int i = 0; i < C::SA; i++) {
            mbar_init(bar(B_AF + i), C::DEC);
            mbar_init(bar(B_AE + i), 1);
        }
        for (int i = 0; i < TC_NB; i++) {
            mbar_init(bar(B_BF + i), 1);
            mbar_init(bar(B_BE + i), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_ACCF + i), 1);
            mbar_init(bar(B_ACCE + i), 4);
        }
        mbar_init(bar(B_FIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (KD == 1) {
        // e4m3 of E2M1 magnitude m times 2^(e-127), for every scale byte e:
        // exact for e in [119, 133]; 255 (a dropped group) and the bytes a
        // layer on this path never holds get zeros.
        uint2 *lut = (uint2 *)(sm + C::LUT_OFF);
        for (int e = threadIdx.x; e < 256; e += blockDim.x) {
            uint32_t t[2] = {0u, 0u};
            if (e >= 119 && e <= 133) {
                const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
#pragma unroll
                for (int m = 1; m < 8; m++)
                    t[m >> 2] |= (uint32_t)__nv_cvt_float_to_fp8(ldexpf(mag[m], e - 127), __NV_SATFINITE, __NV_E4M3)
                                 << (8 * (m & 3));
            }
            lut[e] = make_uint2(t[0], t[1]);
        }
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(TC_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)tmem_slot;

    auto a_stage = [&](int s) { return sbase + (uint32_t)(s * C::A_BYTES); };
    auto pk_stage = [&](int s) { return sbase + (uint32_t)(C::PK_OFF + s * C::PK_BYTES); };
    const uint32_t b_ring = sbase + (uint32_t)C::B_OFF;

    if (warp == W_PK) {
        // ------------------------------------------------ packed weight tiles
        uint32_t it = 0;
        uint32_t issued[C::SP];
#pragma unroll
        for (int i = 0; i < C::SP; i++) issued[i] = 0;
        if (lane == 0) {
            TcTile tl_next = tile_at(cid);
            for (int ug = cid; ug < n_groups && !*abort_flag; ug += ncl) {
                const int u = unit_of(ug);
                const TcTile tl = tl_next;
                tl_next = tile_at(ug + ncl);
                const int rb = u % nrb;
                const CUtensorMap *mp = a.maps + 3 * tl.expert + (PH == 0 ? 0 : 2);
                bool ok = true;
                for (int ss = 0; ss < nss; ss++, it++) {
                    const int slot = it % C::SP;
                    if (it >= (uint32_t)C::SP &&
                        !tc_wait(bar(B_PKE + slot), ((it / C::SP) - 1) & 1, a.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B_PKF + slot), C::PK_BYTES);
                    issued[slot]++;
#pragma unroll
                    for (int m = 0; m < C::NA; m++)
                        tma_load_2d(pk_stage(slot) + (uint32_t)(m * TC_M * 128), mp + m, ss * 128, rb * TC_M,
                                    bar(B_PKF + slot));
                }
                if (!ok) break;
            }
            // drain: every fill issued here has landed before the CTA exits
            for (int s = 0; s < C::SP; s++)
                if (issued[s]) mbar_wait(bar(B_PKF + s), (issued[s] - 1) & 1, a.err);
        }
        __syncwarp();
    } else if (warp == W_B) {
        // --------------------------------------------------- token tiles
        // Slots are counted with free-running counters: a k-step of c slots
        // starts at `head` (skipping to the ring start when it would not fit
        // before the end) and the slots up to the end of the oldest k-step
        // the MMAs have finished are free again.
        if (lane == 0) {
            uint32_t kt = 0, done = 0, head = 0, tail = 0;
            uint32_t endv[TC_NB];
            const int B_FREE = B_BE;
            TcTile tl_next = tile_at(cid);
            for (int ug = cid; ug < n_groups && !*abort_flag; ug += ncl) {
                const TcTile tl = tl_next;
                tl_next = tile_at(ug + ncl);
                const int nb = PH == 0 ? tl.nx : tl.nh;
                if (nb < 16 || nb % 16 || nb > C::BMAX) {
                    set_device_error(a.err, K3MOE_EINVAL);
                    *abort_flag = 1;
                    break;
                }
                // a row holds K elements: e4m3 token rows 1 byte each, bf16 rows 2
                const uint8_t *src = a.Bsrc + (size_t)(PH == 0 ? tl.xrow0 : tl.hrow0) * K * (KD ? 1 : 2);
                const uint32_t bytes = (uint32_t)nb * 128u;
                const uint32_t c = (uint32_t)nb / 16u;
                bool ok = true;
                for (int ks = 0; ks < nks && ok; ks++, kt++) {
                    uint32_t start = head;
                    if (start % C::NSLOT + c > (uint32_t)C::NSLOT) start += C::NSLOT - start % C::NSLOT;
                    while (kt - done >= (uint32_t)TC_NB || start + c - tail > (uint32_t)C::NSLOT) {
                        if (done == kt ||
                            !tc_wait(bar(B_FREE + done % TC_NB), (done / TC_NB) & 1, a.err, abort_flag)) {
                            if (done == kt) set_device_error(a.err, K3MOE_EINVAL);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        tail = endv[done % TC_NB];
                        done++;
                    }
                    if (!ok) break;
                    head = start + c;
                    endv[kt % TC_NB] = head;
                    const uint32_t off = (start % C::NSLOT) * TC_SLOT;
                    boff[kt % TC_NB] = off;
                    mbar_arrive_expect_tx(bar(B_BF + kt % TC_NB), bytes);
                    bulk_g2s(b_ring + off, src + (size_t)ks * bytes, bytes, bar(B_BF + kt % TC_NB));
                }
                if (!ok) break;
            }
            // drain: every copy issued here has landed before the CTA exits
            for (uint32_t q = done; q < kt; q++) mbar_wait(bar(B_BF + q % TC_NB), (q / TC_NB) & 1, a.err);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------ MMA
        // The whole warp walks the loop (the MMAs need a converged warp for
        // elect.sync); every lane takes the same branches.
        uint32_t kt = 0, ut = 0;
        TcTile tl_next = tile_at(cid);
        for (int ug = cid; ug < n_groups && !*abort_flag; ug += ncl, ut++) {
            const TcTile tl = tl_next;
            tl_next = tile_at(ug + ncl);
            const int nb = PH == 0 ? tl.nx : tl.nh;
            if (nb < 16 || nb % 16 || nb > C::BMAX) {
                if (lane == 0) set_device_error(a.err, K3MOE_EINVAL);
                *abort_flag = 1;
                break;
            }
            const uint32_t idesc = KD ? e4m3_idesc(nb) : bf16_idesc(nb);
            const int buf = ut & 1;
            if (ut >= 2 && !__all_sync(0xffffffffu, tc_wait(bar(B_ACCE + buf), ((ut / 2) - 1) & 1, a.err, abort_flag)))
                break;
            tc_fence_after();
            const uint32_t td = tmem + (uint32_t)(buf * 256);
            bool ok = true;
            for (int ks = 0; ks < nks; ks++, kt++) {
                const int sa = kt % C::SA, sb = kt % TC_NB;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_AF + sa), (kt / C::SA) & 1, a.err, abort_flag) &&
                                                 tc_wait(bar(B_BF + sb), (kt / TC_NB) & 1, a.err, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t blo = sw128_lo(b_ring + boff[sb]);
                const uint32_t alo = sw128_lo(a_stage(sa));
                mma_kstep<C::NA, KD>(td, alo, blo, idesc, ks != 0);
                mma_commit(bar(B_AE + sa));
                mma_commit(bar(B_BE + sb));
            }
            if (!ok) break;
            mma_commit(bar(B_ACCF + buf));
        }
        // every MMA issued above has completed before TMEM is freed
        mma_commit(bar(B_FIN));
        mbar_wait(bar(B_FIN), 0, a.err);
        __syncwarp();
    } else if (warp < W_EPI) {
        // ------------------------------------------------------- decoders
        // Thread (row r, part p) decodes IPP of the row's NA x GPK 32-groups
        // of every k-step (items p*IPP .. p*IPP+IPP-1; item = GPK * matrix +
        // group); the items of a part share one matrix.
        const int dw = warp - W_DEC;
        const int r = (dw & 3) * 32 + lane;  // weight row within the unit
        const int part = dw >> 2;
        const int mat = (part * C::IPP) / C::GPK;
        const uint32_t lut = sbase + (uint32_t)C::LUT_OFF;
        uint32_t it = 0, kt = 0;
        const int g_per_ss = TC_SS / 32;  // 8 scale bytes per row per staging step
        auto scale_plane = [&](int e) -> const uint8_t * {
            return PH == 1 ? a.table[e].ds : (mat == 0 ? a.table[e].gs : a.table[e].us);
        };
        // The scale row of the next unit is found in three steps spread over
        // the current unit (its expert at the first staging step, the plane at
        // the middle one, the first 8 bytes at the last one), so no load in the
        // loop waits on another.
        int ug = cid;
        const uint8_t *scl = nullptr, *nplane = nullptr, *nscl = nullptr;
        int nexp = 0;
        if (ug < n_groups)
            scl = scale_plane(a.tiles[ug / gpt].expert) + (size_t)((unit_of(ug) % nrb) * TC_M + r) * (K / 32);
        uint2 sc_next = scl ? __ldg((const uint2 *)scl) : make_uint2(0, 0);
        int ss = 0;
        while (ug < n_groups && !*abort_flag) {
            const int ugn = ug + ncl;
            if (ss == 0 && ugn < n_groups) nexp = a.tiles[ugn / gpt].expert;
            if (ss == nss / 2 && ugn < n_groups) nplane = scale_plane(nexp);
            const uint2 sc = sc_next;
            if (ss + 1 < nss) {
                sc_next = __ldg((const uint2 *)(scl + (ss + 1) * g_per_ss));
            } else if (ugn < n_groups) {
                nscl = nplane + (size_t)((unit_of(ugn) % nrb) * TC_M + r) * (K / 32);
                sc_next = __ldg((const uint2 *)nscl);
            }
            int ss2 = ss + 1, ug2 = ug;
            if (ss2 == nss) {
                ss2 = 0;
                ug2 = ugn;
            }
            const int pslot = it % C::SP;
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_PKF + pslot), (it / C::SP) & 1, a.err, abort_flag))) break;
            bool ok = true;
            for (int kk = 0; kk < C::KPS; kk++, kt++) {
                const int slot = kt % C::SA;
                if (kt >= (uint32_t)C::SA &&
                    !__all_sync(0xffffffffu, tc_wait(bar(B_AE + slot), ((kt / C::SA) - 1) & 1, a.err, abort_flag))) {
                    ok = false;
                    break;
                }
                const uint32_t src = pk_stage(pslot) + (uint32_t)(mat * TC_M * 128 + r * 128);
                const uint32_t dst = a_stage(slot) + (uint32_t)(mat * TC_M * 128 + r * 128);
#pragma unroll
                for (int gg = 0; gg < C::IPP; gg++) {
                    const int g = (part * C::IPP + gg) % C::GPK;  // 32-group within the k-step
                    // the group's 16 packed bytes are chunk pc of the staged row, its
                    // scale byte pc of the staging step's 8
                    const int pc = kk * C::GPK + g;
                    const uint4 q = lds128(src + (uint32_t)((pc ^ (r & 7)) << 4));
                    const uint32_t e = ((pc < 4 ? sc.x : sc.y) >> (8 * (pc & 3))) & 0xffu;
                    if constexpr (KD == 1) {
                        const uint2 t = lds64(lut + e * 8);
                        const uint2 o0 = decode8_e4m3(q.x, t.x, t.y), o1 = decode8_e4m3(q.y, t.x, t.y);
                        const uint2 o2 = decode8_e4m3(q.z, t.x, t.y), o3 = decode8_e4m3(q.w, t.x, t.y);
                        // 32 e4m3 bytes = chunks 2g and 2g + 1 of the k-step's 128-byte row
                        const uint32_t a0 = dst + (uint32_t)((((2 * g) ^ (r & 7))) << 4);
                        const uint32_t a1 = dst + (uint32_t)((((2 * g + 1) ^ (r & 7))) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(o0.x), "r"(o0.y),
                                     "r"(o1.x), "r"(o1.y)
                                     : "memory");
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(o2.x), "r"(o2.y),
                                     "r"(o3.x), "r"(o3.y)
                                     : "memory");
                        continue;
                    }
                    bool fast;
                    const uint16_t sh = e8m0_f16(e, fast);
                    uint4 o[4];
                    if (__all_sync(0xffffffffu, fast)) {
                        o[0] = decode8_bf16(q.x, sh);
                        o[1] = decode8_bf16(q.y, sh);
                        o[2] = decode8_bf16(q.z, sh);
                        o[3] = decode8_bf16(q.w, sh);
                    } else {
                        const float sf = e8m0_scale(e);
                        o[0] = decode8_bf16_any(q.x, sf);
                        o[1] = decode8_bf16_any(q.y, sf);
                        o[2] = decode8_bf16_any(q.z, sf);
                        o[3] = decode8_bf16_any(q.w, sf);
                    }
#pragma unroll
                    for (int w = 0; w < 4; w++) {
                        const int c = g * 4 + w;  // 16-byte chunk of the k-step's 128-byte bf16 row
                        const uint32_t ad = dst + (uint32_t)(((c ^ (r & 7)) << 4));
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ad), "r"(o[w].x), "r"(o[w].y),
                                     "r"(o[w].z), "r"(o[w].w)
                                     : "memory");
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_AF + slot));
            }
            if (!ok) break;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PKE + pslot));
            it++;
            if (ug2 != ug) scl = nscl;
            ug = ug2;
            ss = ss2;
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;       // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;  // weight row within the unit
        uint32_t ut = 0;
        TcTile tl_next = tile_at(cid);
        for (int ug = cid; ug < n_groups && !*abort_flag; ug += ncl, ut++) {
            const int u = unit_of(ug);
            const TcTile tl = tl_next;
            tl_next = tile_at(ug + ncl);
            const int buf = ut & 1;
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_ACCF + buf), (ut / 2) & 1, a.err, abort_flag))) break;
            tc_fence_after();
            const int rb = u % nrb;
            const int P = tile_p(tl.n);
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 256);
            // token pieces: columns c P + j, piece c weighing rho^c (rho = 1 for
            // bf16 hi/lo, 1/16 for e4m3 pieces, which also carry the token's
            // scale); summed from the smallest piece up
            const int np = tl.split > 1 ? tl.split : 1;
            const float rho = KD ? 0.0625f : 1.0f;
            for (int j0 = 0; j0 < tl.n; j0 += 8) {
                if (PH == 0) {
                    float g[8], v[8], t[8];
                    tmem_ld8(tbase + (np - 1) * P + j0, g);
                    tmem_ld8(tbase + 128 + (np - 1) * P + j0, v);
                    tmem_wait_ld();
                    for (int c = np - 2; c >= 0; c--) {
                        tmem_ld8(tbase + c * P + j0, t);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; i++) g[i] = fmaf(g[i], rho, t[i]);
                        tmem_ld8(tbase + 128 + c * P + j0, t);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; i++) v[i] = fmaf(v[i], rho, t[i]);
                    }
                    if (KD == 1) {
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const int j = min(j0 + i, tl.n - 1);
                            const float sx = a.tscale[a.perm[tl.pair_begin + j] / a.k];
                            g[i] *= sx;
                            v[i] *= sx;
                        }
                    }
                    const int col = rb * TC_M + r;  // index into f
                    if (a.hf) {
                        // e4m3 down: h in fp32 and its per-pair maximum magnitude
#pragma unroll
                        for (int jj = 0; jj < 8; jj++) {
                            const int j = j0 + jj;
                            if (j < tl.n) {
                                const float h = silu(g[jj]) * v[jj];
                                a.hf[(size_t)(tl.pair_begin + j) * a.f + col] = h;
                                float m = fabsf(h);
#pragma unroll
                                for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                                if (lane == 0) atomicMax(a.hmax + tl.pair_begin + j, __float_as_uint(m));
                            }
                        }
                        continue;
                    }
                    const int s = col >> 6, c = (col & 63) >> 3, byte = (col & 7) * 2;
                    uint8_t *hb = a.Hg + (size_t)tl.hrow0 * a.f * 2 + (size_t)s * tl.nh * 128 + byte;
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        const int j = j0 + jj;
                        if (j < tl.n) {
                            const float h = silu(g[jj]) * v[jj];
                            const uint32_t hi = bf16_rn_bits(h);
                            const uint32_t lo = bf16_rn_bits(h - __uint_as_float(hi << 16));
                            const int jh = j, jl = P + j;
                            *(uint16_t *)(hb + jh * 128 + ((c ^ (jh & 7)) << 4)) = (uint16_t)hi;
                            *(uint16_t *)(hb + jl * 128 + ((c ^ (jl & 7)) << 4)) = (uint16_t)lo;
                        }
                    }
                } else {
                    // h pieces: bf16 hi, lo (rho = 1) or four e4m3 pieces (rho =
                    // 1/16, times the pair's h scale)
                    const int nph = KD ? 4 : 2;
                    float y[8], t[8];
                    tmem_ld8(tbase + (nph - 1) * P + j0, y);
                    tmem_wait_ld();
                    for (int c = nph - 2; c >= 0; c--) {
                        tmem_ld8(tbase + c * P + j0, t);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 8; i++) y[i] = fmaf(y[i], rho, t[i]);
                    }
                    // lane l of group q (rows 8q..8q+7 of this warp's 32) now takes
                    // token j0 + (l & 7) of the eight and adds its eight rows with
                    // two vector reductions instead of eight scalar atomics
                    transpose8(y, lane);
                    const int j = j0 + (lane & 7);
                    if (j < tl.n) {
                        const int pair = a.perm[tl.pair_begin + j];
                        float w = a.wsel[pair];
                        if (KD == 1) w *= h_scale(a.hmax[tl.pair_begin + j]);
                        float *o = a.out + (size_t)(pair / a.k) * a.d + rb * TC_M + q * 32 + (lane & ~7);
                        red_add_v4(o, w * y[0], w * y[1], w * y[2], w * y[3]);
                        red_add_v4(o + 4, w * y[4], w * y[5], w * y[6], w * y[7]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_ACCE + buf));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- planning

// Tiles of at most tn tokens per expert, with the row offsets of each tile in
// the token array (nx rows) and in the h array (nh rows).  One CTA.
__global__ void __launch_bounds__(1024) k3_tc_plan(const int32_t *__restrict__ offsets, int E, int tn,
                                                   int np, int nph, int max_tiles, TcTile *tiles,
                                                   int32_t *n_tiles, int *err)
{
    __shared__ int wsum[3][32];
    __shared__ int base[3];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) base[0] = base[1] = base[2] = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int c = e < E ? offsets[e + 1] - offsets[e] : 0;
        const int nt = (c + tn - 1) / tn;
        int rx = 0, rh = 0;
        for (int j = 0; j < nt; j++) {
            const int n = min(tn, c - j * tn);
            rx += tile_nx(n, np);
            rh += tile_nh(n, nph);
        }
        int v[3] = {nt, rx, rh}, inc[3];
#pragma unroll
        for (int i = 0; i < 3; i++) {
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
            for (int i = 0; i < 3; i++) {
                int x = lane < nw ? wsum[i][lane] : 0;
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane < nw) wsum[i][lane] = x - wsum[i][lane];  // exclusive
            }
        }
        __syncthreads();
        int t = base[0] + wsum[0][warp] + inc[0] - v[0];
        int xr = base[1] + wsum[1][warp] + inc[1] - v[1];
        int hr = base[2] + wsum[2][warp] + inc[2] - v[2];
        for (int j = 0; j < nt; j++, t++) {
            const int n = min(tn, c - j * tn);
            const int nx = tile_nx(n, np), nh = tile_nh(n, nph);
            if (t < max_tiles) {
                TcTile tl;
                tl.expert = e;
                tl.pair_begin = offsets[e] + j * tn;
                tl.n = n;
                tl.nx = nx;
                tl.nh = nh;
                tl.xrow0 = xr;
                tl.hrow0 = hr;
                tl.split = np;
                tiles[t] = tl;
            }
            xr += nx;
            hr += nh;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {
            base[0] = t;
            base[1] = xr;
            base[2] = hr;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (base[0] > max_tiles) {
            set_device_error(err, K3MOE_EINVAL);
            *n_tiles = 0;
        } else {
            *n_tiles = base[0];
        }
    }
}

// Token rows of every tile, k-step-major and pre-swizzled: the 8 16-byte
// chunks of a row's 128-byte k-step slice sit at chunk ^ (row & 7).
// KD = 0: bf16 rows (fp32 tokens as hi, lo pieces).  KD = 1: e4m3 pieces,
// piece c = RN(r_c / s_c) with r_0 = x, r_{c+1} = r_c - s_c * piece c and
// s_c = s_0 16^-c (s_0 = the token's scale, a power of two): every step is
// exact in fp32, so the pieces sum to x within s_0 16^-np.
template <typename XT, int KD>
__global__ void __launch_bounds__(256) k3_tc_gather(const XT *__restrict__ X, const int32_t *__restrict__ perm,
                                                    int k, int d, const TcTile *__restrict__ tiles,
                                                    const int32_t *n_tiles, const float *__restrict__ tscale,
                                                    uint8_t *Xg)
{
    // One thread per (token of the tile, 16-byte output chunk): the token's
    // elements are read once and all its pieces written.  Rows past n (the
    // padding of each piece) are left as they are: they only feed MMA
    // columns that no epilogue reads.
    const int nt = *n_tiles;
    const int EPC = KD ? 16 : 8;  // elements per 16-byte chunk
    const int cpr = d / EPC;      // chunks per row
    const size_t rowb = KD ? (size_t)d : (size_t)d * 2;
    for (int t = blockIdx.x; t < nt; t += gridDim.x) {
        const TcTile tl = tiles[t];
        const int P = tile_p(tl.n);
        const int np = tl.split > 1 ? tl.split : 1;
        uint8_t *base = Xg + (size_t)tl.xrow0 * rowb;
        for (int idx = threadIdx.x; idx < tl.n * cpr; idx += blockDim.x) {
            const int j = idx / cpr, ch = idx - j * cpr;
            const int s = ch >> 3, c = ch & 7;
            const int tok = perm[tl.pair_begin + j] / k;
            float v[16];
            if constexpr (sizeof(XT) == 2) {
                const uint4 *src = (const uint4 *)((const uint16_t *)X + (size_t)tok * d + ch * EPC);
#pragma unroll
                for (int q = 0; q < EPC / 8; q++) {
                    const uint4 u = src[q];
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
                        v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                    }
                }
            } else {
                const float4 *src = (const float4 *)((const float *)X + (size_t)tok * d + ch * EPC);
#pragma unroll
                for (int q = 0; q < EPC / 4; q++) {
                    const float4 f4 = src[q];
                    v[4 * q] = f4.x;
                    v[4 * q + 1] = f4.y;
                    v[4 * q + 2] = f4.z;
                    v[4 * q + 3] = f4.w;
                }
            }
            auto put = [&](int piece, uint4 o) {
                const int row = piece * P + j;
                *(uint4 *)(base + (size_t)s * tl.nx * 128 + row * 128 + ((c ^ (row & 7)) << 4)) = o;
            };
            if constexpr (KD == 0) {
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    hi[i] = bf16_rn_bits(v[i]);
                    lo[i] = bf16_rn_bits(v[i] - __uint_as_float(hi[i] << 16));
                }
                put(0, make_uint4(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16), hi[4] | (hi[5] << 16),
                                  hi[6] | (hi[7] << 16)));
                if (np > 1)
                    put(1, make_uint4(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16), lo[4] | (lo[5] << 16),
                                      lo[6] | (lo[7] << 16)));
            } else {
                const float inv0 = 1.0f / tscale[tok];  // a power of two: exact
#pragma unroll
                for (int i = 0; i < 16; i++) v[i] *= inv0;  // in units of s_0
                for (int piece = 0; piece < np; piece++) {
                    uint32_t b[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int i = 0; i < 16; i += 2) {
                        const uint32_t q2 =
                            __nv_cvt_float2_to_fp8x2(make_float2(v[i], v[i + 1]), __NV_SATFINITE, __NV_E4M3);
                        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)q2, __NV_E4M3);
                        const float2 back = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                        v[i] = (v[i] - back.x) * 16.0f;
                        v[i + 1] = (v[i + 1] - back.y) * 16.0f;
                        b[i >> 2] |= (q2 & 0xffffu) << (8 * (i & 3));  // elements i, i + 1 -> bytes i, i + 1
                    }
                    put(piece, make_uint4(b[0], b[1], b[2], b[3]));
                }
            }
        }
    }
}

// h rows of every tile as four e4m3 pieces (rows c P + j, k-step-major,
// pre-swizzled like the token rows), from h in fp32 and the pair's scale.
__global__ void __launch_bounds__(256) k3_tc_hpieces(const float *__restrict__ hf, const unsigned *__restrict__ hmax,
                                                    int f, const TcTile *__restrict__ tiles, const int32_t *n_tiles,
                                                    uint8_t *Hg)
{
    const int nt = *n_tiles;
    const int cpr = f / 16;  // 16-element chunks per row
    for (int t = blockIdx.x; t < nt; t += gridDim.x) {
        const TcTile tl = tiles[t];
        const int P = tile_p(tl.n);
        uint8_t *base = Hg + (size_t)tl.hrow0 * f;
        for (int idx = threadIdx.x; idx < tl.n * cpr; idx += blockDim.x) {
            const int j = idx / cpr, ch = idx - j * cpr;
            const int s = ch >> 3, c = ch & 7;
            const float inv0 = 1.0f / h_scale(hmax[tl.pair_begin + j]);  // a power of two: exact
            const float4 *src = (const float4 *)(hf + (size_t)(tl.pair_begin + j) * f + ch * 16);
            float r[16];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 v = src[q];
                r[4 * q] = v.x * inv0;
                r[4 * q + 1] = v.y * inv0;
                r[4 * q + 2] = v.z * inv0;
                r[4 * q + 3] = v.w * inv0;
            }
#pragma unroll
            for (int piece = 0; piece < 4; piece++) {
                uint32_t b[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const uint32_t q2 =
                        __nv_cvt_float2_to_fp8x2(make_float2(r[i], r[i + 1]), __NV_SATFINITE, __NV_E4M3);
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)q2, __NV_E4M3);
                    const float2 back = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                    r[i] = (r[i] - back.x) * 16.0f;
                    r[i + 1] = (r[i + 1] - back.y) * 16.0f;
                    b[i >> 2] |= (q2 & 0xffffu) << (8 * (i & 3));
                }
                const int row = piece * P + j;
                *(uint4 *)(base + (size_t)s * tl.nh * 128 + row * 128 + ((c ^ (row & 7)) << 4)) =
                    make_uint4(b[0], b[1], b[2], b[3]);
            }
        }
    }
}

// s_0 of every token for e4m3 pieces: 2^(x - 8) where the token's largest
// magnitude is m 2^x, m in [0.5, 1), so that |x| / s_0 < 256 < 448 (the e4m3
// maximum); 1 for an all-zero token.  One warp per token.
template <typename XT>
__global__ void __launch_bounds__(256) k3_tc_token_scale(const XT *__restrict__ X, int T, int d, float *tscale)
{
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    float m = 0.f;
    for (int i = lane; i < d; i += 32) {
        float v;
        if constexpr (sizeof(XT) == 2)
            v = __uint_as_float((uint32_t)((const uint16_t *)X)[(size_t)t * d + i] << 16);
        else
            v = ((const float *)X)[(size_t)t * d + i];
        m = fmaxf(m, fabsf(v));
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    if (lane == 0) tscale[t] = piece_scale(m);
}

// Counts the scale bytes of every expert (gate, up, down) outside [119, 133] and
// other than 255 (the bytes the e4m3 decode cannot represent exactly).
__global__ void __launch_bounds__(256) k3_tc_scale_range(const DevExpert *__restrict__ table, int E, int d, int f,
                                                        unsigned *bad)
{
    const int e = blockIdx.x, m = blockIdx.y;
    const uint8_t *p = m == 0 ? table[e].gs : m == 1 ? table[e].us : table[e].ds;
    const size_t n = m < 2 ? (size_t)f * (d / 32) : (size_t)d * (f / 32);
    unsigned cnt = 0;
    for (size_t i = threadIdx.x * 16; i < n; i += blockDim.x * 16) {
        const uint4 q = *(const uint4 *)(p + i);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const uint32_t b = (w[j >> 2] >> (8 * (j & 3))) & 0xffu;
            cnt += (b != 255u && (b < 119u || b > 133u));
        }
    }
    if (cnt) atomicAdd(bad, cnt);
}

// ------------------------------------------------------------------ router

// logits[t][e] = sum_i X[t][i] W_r[e][i] for bf16 tokens on the tensor cores:
// one CTA per (128 experts x 256 tokens) tile, both operands by TMA (128-byte
// swizzle, out-of-range rows read as zeros), fp32 accumulation in TMEM.
// bf16 x bf16 products are exact in fp32.  Warp 0: TMA; warp 1: MMA; warps
// 2-5: epilogue.
constexpr int RT_S = 4, RT_N = 256, RT_A = TC_M * 128, RT_B = RT_N * 128;
constexpr int RT_SMEM = RT_S * (RT_A + RT_B) + 256 + 1024;

__global__ void __launch_bounds__(192, 1) k3_router_tc(const __grid_constant__ CUtensorMap wmap,
                                                      const __grid_constant__ CUtensorMap xmap, int T, int E, int d,
                                                      float *logits, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(sm);
    uint64_t *bars = (uint64_t *)(sm + RT_S * (RT_A + RT_B));
    const int B_F = 0, B_E = RT_S, B_ACC = 2 * RT_S, B_FIN = 2 * RT_S + 1;
    uint32_t *tmem_slot = (uint32_t *)(bars + B_FIN + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * TC_M, n0 = blockIdx.y * RT_N, nks = d / 64;
    if (threadIdx.x == 0) {
        for (int i = 0; i < RT_S; i++) {
            mbar_init(bar(B_F + i), 1);
            mbar_init(bar(B_E + i), 1);
        }
        mbar_init(bar(B_ACC), 1);
        mbar_init(bar(B_FIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(RT_N)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)tmem_slot;
    auto stage = [&](int s) { return sbase + (uint32_t)(s * (RT_A + RT_B)); };
    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int ks = 0; ks < nks && !*abort_flag; ks++, issued++) {
                const int s = ks % RT_S;
                if (ks >= RT_S && !tc_wait(bar(B_E + s), ((ks / RT_S) - 1) & 1, err, abort_flag)) break;
                mbar_arrive_expect_tx(bar(B_F + s), RT_A + RT_B);
                asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
                             "[%1, {%2, %3}], [%4];" ::"r"(stage(s)),
                             "l"((uint64_t)&wmap), "r"(ks * 64), "r"(m0), "r"(bar(B_F + s))
                             : "memory");
                asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
                             "[%1, {%2, %3}], [%4];" ::"r"(stage(s) + RT_A),
                             "l"((uint64_t)&xmap), "r"(ks * 64), "r"(n0), "r"(bar(B_F + s))
                             : "memory");
            }
            for (int q = issued > RT_S ? issued - RT_S : 0; q < issued; q++)  // drain
                mbar_wait(bar(B_F + q % RT_S), (q / RT_S) & 1, err);
        }
        __syncwarp();
    } else if (warp == 1) {
        const uint32_t idesc = bf16_idesc(RT_N);
        bool ok = true;
        for (int ks = 0; ks < nks && !*abort_flag; ks++) {
            const int s = ks % RT_S;
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_F + s), (ks / RT_S) & 1, err, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            mma_kstep<1, 0>(tmem, sw128_lo(stage(s)), sw128_lo(stage(s) + RT_A), idesc, ks != 0);
            mma_commit(bar(B_E + s));
        }
        if (ok) mma_commit(bar(B_ACC));
        mma_commit(bar(B_FIN));
        mbar_wait(bar(B_FIN), 0, err);
        __syncwarp();
    } else {
        const int q = warp & 3;
        if (__all_sync(0xffffffffu, tc_wait(bar(B_ACC), 0, err, abort_flag))) {
            tc_fence_after();
            const int e = m0 + q * 32 + lane;
            for (int c0 = 0; c0 < RT_N; c0 += 8) {
                float v[8];
                tmem_ld8(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int t = n0 + c0 + i;
                    if (e < E && t < T) logits[(size_t)t * E + e] = v[i];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(RT_N) : "memory");
    }
}

// --------------------------------------------------------------- launchers

int num_sms();

bool tc_supported(int E, int k, int d, int f)
{
    return E >= 1 && k >= 1 && d % TC_SS == 0 && f % TC_SS == 0 && d >= TC_SS && f >= TC_SS &&
           d <= 16384 && f <= 16384;
}
// Tokens per tile and pieces per token row for each operand kind: every
// gate/up MMA is at most 128 columns wide.
int tc_tile_tokens(int xdt, int kd) { return kd ? (xdt == K3MOE_BF16 ? 64 : 32) : (xdt == K3MOE_BF16 ? 128 : 64); }
static int tc_pieces(int xdt, int kd) { return kd ? (xdt == K3MOE_BF16 ? 2 : 4) : (xdt == K3MOE_BF16 ? 1 : 2); }
int tc_max_tiles(int npairs, int E) { return (npairs + 31) / 32 + E; }
// Bytes of the token and h row arrays, the worst case over kinds and types.
size_t tc_xg_bytes(int npairs, int E, int d) { return 4 * ((size_t)npairs + 7 * (size_t)tc_max_tiles(npairs, E)) * d; }
size_t tc_hg_bytes(int npairs, int E, int f) { return 2 * ((size_t)npairs + 7 * (size_t)tc_max_tiles(npairs, E)) * f * 2; }
size_t tc_tile_bytes() { return sizeof(TcTile); }
size_t tc_map_bytes() { return sizeof(CUtensorMap); }

// 1 when every scale byte of the E experts is in [119, 133] or 255 (the e4m3
// decode is exact), 0 otherwise, negative on error.
int tc_e4m3_eligible(const DevExpert *dev_table, int E, int d, int f, cudaStream_t s)
{
    unsigned *bad = nullptr;
    unsigned h = 1;
    if (cudaMalloc(&bad, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ENOMEM;
    }
    int rc = K3MOE_OK;
    if (cudaMemsetAsync(bad, 0, sizeof(unsigned), s) != cudaSuccess) rc = K3MOE_ECUDA;
    if (rc == K3MOE_OK) {
        k3_tc_scale_range<<<dim3(E, 3), 256, 0, s>>>(dev_table, E, d, f, bad);
        if (cudaGetLastError() != cudaSuccess ||
            cudaMemcpyAsync(&h, bad, sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            rc = K3MOE_ECUDA;
    }
    cudaGetLastError();
    cudaFree(bad);
    return rc == K3MOE_OK ? (h == 0 ? 1 : 0) : rc;
}

// Tensor maps of the packed planes of E experts (host table of device plane
// pointers): [E][gate, up, down], 2D u8 tensors of rows x in/2 bytes, boxes
// of 128 rows x 128 bytes with the 128-byte swizzle, written to dev_maps.
int tc_make_maps(const DevExpert *host_table, int E, int d, int f, void *dev_maps)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return K3MOE_ECUDA;
        }
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    CUtensorMap *maps = (CUtensorMap *)malloc(sizeof(CUtensorMap) * 3 * (size_t)E);
    if (!maps) return K3MOE_ENOMEM;
    int rc = K3MOE_OK;
    for (int e = 0; e < E && rc == K3MOE_OK; e++) {
        const uint8_t *planes[3] = {host_table[e].gp, host_table[e].up, host_table[e].dp};
        for (int m = 0; m < 3; m++) {
            const int rows = m < 2 ? f : d, in = m < 2 ? d : f;
            const cuuint64_t dims[2] = {(cuuint64_t)(in / 2), (cuuint64_t)rows};
            const cuuint64_t strides[1] = {(cuuint64_t)(in / 2)};
            const cuuint32_t box[2] = {128, (cuuint32_t)TC_M};
            const cuuint32_t estr[2] = {1, 1};
            if (encode(&maps[3 * e + m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void *)planes[m], dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
                rc = K3MOE_EINVAL;
                break;
            }
        }
    }
    if (rc == K3MOE_OK &&
        cudaMemcpy(dev_maps, maps, sizeof(CUtensorMap) * 3 * (size_t)E, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        rc = K3MOE_ECUDA;
    }
    free(maps);
    return rc;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return nullptr;
        }
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    return encode;
}

// Router logits of bf16 tokens on the tensor cores (see k3_router_tc):
// logits [T x E] fp32.  Needs d % 64 == 0.
int launch_router_tc(const uint16_t *X, int T, const uint16_t *Wr, int E, int d, float *logits, int *err,
                     cudaStream_t s)
{
    auto encode = tensor_map_encoder();
    if (!encode || d % 64) return K3MOE_ECUDA;
    CUtensorMap wmap, xmap;
    const cuuint64_t wdims[2] = {(cuuint64_t)d, (cuuint64_t)E}, xdims[2] = {(cuuint64_t)d, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t wbox[2] = {64, (cuuint32_t)TC_M}, xbox[2] = {64, (cuuint32_t)RT_N}, es[2] = {1, 1};
    if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)Wr, wdims, strides, wbox, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void *)X, xdims, strides, xbox, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return K3MOE_EINVAL;
    if (ensure_smem((const void *)k3_router_tc, RT_SMEM) != K3MOE_OK) return K3MOE_ECUDA;
    const dim3 grid((E + TC_M - 1) / TC_M, (T + RT_N - 1) / RT_N);
    k3_router_tc<<<grid, 192, RT_SMEM, s>>>(wmap, xmap, T, E, d, logits, err);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

// Launches one phase on persistent CTAs, one per SM.
template <int PH, int KD>
static int launch_expert(const TcArgs &a, cudaStream_t s)
{
    using C = TcCfg<PH, KD>;
    if (ensure_smem((const void *)k3_tc_expert<PH, KD>, C::SMEM) != K3MOE_OK) return K3MOE_ECUDA;
    k3_tc_expert<PH, KD><<<num_sms(), C::THREADS, C::SMEM, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    return K3MOE_OK;
}

// Plan, token rows and the gate/up + SwiGLU phase (h into Hg); kd = 1 runs
// gate/up on e4m3 operands (only for layers whose scale bytes allow it).
int launch_tc_gateup(const void *X, int xdt, int T, int kd, int k, int E, int d, int f, const DevExpert *table,
                     const void *maps, const int32_t *offsets, const int32_t *perm, void *tiles, int32_t *n_tiles,
                     int max_tiles, float *tscale, uint8_t *Xg, uint8_t *Hg, float *hf, unsigned *hmax, int *err,
                     cudaStream_t s)
{
    const int tn = tc_tile_tokens(xdt, kd), np = tc_pieces(xdt, kd);
    k3_tc_plan<<<1, 1024, 0, s>>>(offsets, E, tn, np, kd ? 4 : 2, max_tiles, (TcTile *)tiles, n_tiles, err);
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    if (kd) {
        if (cudaMemsetAsync(hmax, 0, sizeof(unsigned) * (size_t)T * k, s) != cudaSuccess) return K3MOE_ECUDA;
        if (xdt == K3MOE_BF16)
            k3_tc_token_scale<uint16_t><<<(T + 7) / 8, 256, 0, s>>>((const uint16_t *)X, T, d, tscale);
        else
            k3_tc_token_scale<float><<<(T + 7) / 8, 256, 0, s>>>((const float *)X, T, d, tscale);
        if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    }
    const int g = 2 * num_sms();
    const TcTile *tl = (const TcTile *)tiles;
    if (xdt == K3MOE_BF16) {
        if (kd)
            k3_tc_gather<uint16_t, 1><<<g, 256, 0, s>>>((const uint16_t *)X, perm, k, d, tl, n_tiles, tscale, Xg);
        else
            k3_tc_gather<uint16_t, 0><<<g, 256, 0, s>>>((const uint16_t *)X, perm, k, d, tl, n_tiles, tscale, Xg);
    } else {
        if (kd)
            k3_tc_gather<float, 1><<<g, 256, 0, s>>>((const float *)X, perm, k, d, tl, n_tiles, tscale, Xg);
        else
            k3_tc_gather<float, 0><<<g, 256, 0, s>>>((const float *)X, perm, k, d, tl, n_tiles, tscale, Xg);
    }
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    TcArgs a = {};
    a.tiles = tl;
    a.n_tiles = n_tiles;
    a.table = table;
    a.maps = (const CUtensorMap *)maps;
    a.Bsrc = Xg;
    a.Hg = Hg;
    a.perm = perm;
    a.tscale = tscale;
    a.hf = kd ? hf : nullptr;
    a.hmax = hmax;
    a.k = k;
    a.d = d;
    a.f = f;
    a.err = err;
    return kd ? launch_expert<0, 1>(a, s) : launch_expert<0, 0>(a, s);
}

// Down phase and the weighted combine: out = sum_j w_j y_j (out is zeroed first).
int launch_tc_down(int T, int kd, int k, int d, int f, const DevExpert *table, const void *maps, const int32_t *perm,
                   const float *wsel, const void *tiles, const int32_t *n_tiles, uint8_t *Hg, const float *hf,
                   unsigned *hmax, float *out, int *err, cudaStream_t s)
{
    if (kd) {
        k3_tc_hpieces<<<2 * num_sms(), 256, 0, s>>>(hf, hmax, f, (const TcTile *)tiles, n_tiles, Hg);
        if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    }
    if (cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * d, s) != cudaSuccess) return K3MOE_ECUDA;
    TcArgs a = {};
    a.tiles = (const TcTile *)tiles;
    a.n_tiles = n_tiles;
    a.table = table;
    a.maps = (const CUtensorMap *)maps;
    a.Bsrc = Hg;
    a.out = out;
    a.perm = perm;
    a.wsel = wsel;
    a.hmax = hmax;
    a.k = k;
    a.d = d;
    a.f = f;
    a.err = err;
    return kd ? launch_expert<1, 1>(a, s) : launch_expert<1, 0>(a, s);
}

}  // namespace k3
