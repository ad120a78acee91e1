// k3_mxq.cu -- multi-token expert products with MXFP4 activations on the
// block-scaled tensor cores (tcgen05.mma kind::mxf4, both operands E2M1 with
// one E8M0 scale per 32 along K).
//
// The pages store the expert weights as E2M1 codes with one E8M0 exponent
// per 32 ("kimi-k3-in-c" explainer, "Reduction one: the experts already ship
// at half a byte").  When the activations are quantised to the same format
// (the OCP Microscaling v1.0 conversion: per 32-block the exponent
// floor(log2 amax) - 2, values rounded to the nearest E2M1 magnitude, ties to
// the even code, saturating at 6), a batch's expert products are dense
// block-scaled MXFP4 GEMMs:
//
//   x tiles   k3_mxq_xtiles quantises each token's 32-blocks once and writes
//             the codes and scale bytes into every tile that holds the token
//             (tiles of at most 128 tokens of one expert; k-step-major rows,
//             128-byte swizzled, scale bytes in the 512-byte atoms that
//             tcgen05.cp copies to TMEM)
//   gate/up   k3_mxq_expert<0>: units (tile, 128 rows of f); per 256-long k-step
//             the gate and up weight tiles and their scale boxes by TMA, the
//             tile's token rows and scale atoms by bulk copy, 2 x 4 MMAs of
//             M = 128, N = the tile's tokens, K = 64; the epilogue forms
//             h = silu(g) * u in fp32 and quantises it by the same rule per
//             32 rows of f (one warp's 32 lanes), straight into the down
//             phase's B layout
//   down      k3_mxq_expert<1>: units (tile, 128 rows of d), K = f; the epilogue
//             adds w * y into out with vector reductions
//
// The weights go from HBM to the tensor cores as stored: nothing is decoded.
// Every wait is bounded (2 s); a timeout sets the device error word, the CTA
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "k3_tcgen05.cuh"

namespace k3 {

// One tile: n (<= 128) tokens of one expert, in rows [row0, row0 + np) of the
// token and h row arrays (np = n rounded up to 16, the MMA width).
struct MqTile {
    int32_t expert, pair_begin, n, np, row0, pad0, pad1, pad2;
};

namespace {

constexpr int MQ_M = 128;     // weight rows per unit (MMA M)
constexpr int MQ_TN = 128;    // tokens per tile at most (MMA N <= 128)
constexpr int MQ_THREADS = 256;
constexpr int MQ_W_PROD = 0, MQ_W_MMA = 1, MQ_W_PERM = 2, MQ_W_EPI = 4;

// Instruction descriptor of kind::mxf4 block_scale: E2M1 A and B, K-major,
// N columns, UE8M0 scales, M = 128, the byte of the A and B scale words that
// holds this MMA's first scale.
K3_DEV uint32_t mq_idesc(int n, uint32_t ida, uint32_t idb)
{
    return (idb << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(MQ_M >> 4) << 24) | (ida << 29);
}
K3_DEV void mq_mma(uint32_t td, uint32_t alo, uint32_t blo, uint32_t idesc, uint32_t sfa, uint32_t sfb, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "mov.b64 da, {%1, %7};\n\tmov.b64 db, {%2, %7};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], da, db, %3, [%5], [%6], p;\n\t}"
                 ::"r"(td), "r"(alo), "r"(blo), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb), "r"(SW128_HI)
                 : "memory");
}
// One 512-byte scale atom (32 rows x 16 bytes) from shared memory to TMEM
// columns taddr .. taddr + 3, repeated in the four lane quadrants.
K3_DEV void mq_cp_atom(uint32_t taddr, uint32_t saddr)
{
    const uint32_t lo = ((saddr & 0x3FFFFu) >> 4) | (1u << 16), hi = (128u >> 4) | (1u << 14);
    asm volatile("{\n\t.reg .pred e;\n\t.reg .b64 d;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "mov.b64 d, {%1, %2};\n\t@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], d;\n\t}" ::"r"(taddr),
                 "r"(lo), "r"(hi)
                 : "memory");
}
K3_DEV uint32_t mq_lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
K3_DEV void mq_sts32(uint32_t a, uint32_t v) { asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory"); }
K3_DEV void mq_red_v4(float *out, float v0, float v1, float v2, float v3)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(out), "f"(v0), "f"(v1), "f"(v2), "f"(v3)
                 : "memory");
}
// 8 x 8 transpose within groups of 8 lanes: before, lane g holds
// v[i] = A[g][i]; after, v[i] = A[i][g].
K3_DEV void mq_transpose8(float (&v)[8], int lane)
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

}  // namespace

// Code of |v| (bits ab, sign bit sg) in a block whose largest magnitude has
// bits mb (the rule below); e receives the block's E8M0 byte.
K3_DEV uint32_t mxq_rule(uint32_t ab, uint32_t sg, uint32_t mb, uint32_t &e)
{
    if (mb >= 0x7f800000u) {
        e = 255u;
        return 0u;
    }
    e = (uint32_t)min(max((int)(mb >> 23) - 2, 0), 254);     // floor(log2 amax) - 2 + 127
    const float a = __uint_as_float(ab) * __uint_as_float((254u - e) << 23);  // |v| * 2^(127 - e) < 8, exact
    uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
    return sg ? (c | 8u) : c;
}
// The OCP MX conversion of one 32-block held one value per lane: returns this
// lane's 4-bit code (bit 3 the sign; -0 is code 8) and, in *sbyte, the
// block's E8M0 byte.  A block holding a non-finite value gets byte 255 and
// codes 0.  The exponent is floor(log2 amax) - 2 (the largest E2M1 exponent),
// clamped to [0, 254]; |v| / 2^(e-127) is exact (a power-of-two scaling) and
// rounds to the nearest E2M1 magnitude, ties to the even code, saturating at
// 6.
K3_DEV uint32_t mxq_code(float v, uint32_t *sbyte)
{
    const uint32_t ab = __float_as_uint(v) & 0x7fffffffu;
    const uint32_t mb = __reduce_max_sync(0xffffffffu, ab);  // non-negative floats order like their bits
    uint32_t e;
    const uint32_t c = mxq_rule(ab, __float_as_uint(v) >> 31, mb, e);
    *sbyte = e;
    return c;
}
// The 32 codes of a block packed as 16 bytes (element 2i in the low nibble
// of byte i): word w of the chunk is in lane 8 w after the call.
K3_DEV uint32_t mxq_pack(uint32_t code, int lane)
{
    uint32_t word = code << (4 * (lane & 7));
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    word |= __shfl_xor_sync(0xffffffffu, word, 4);
    return word;
}
// The 16-byte chunk in every lane.
K3_DEV uint4 mxq_chunk(uint32_t word)
{
    return make_uint4(__shfl_sync(0xffffffffu, word, 0), __shfl_sync(0xffffffffu, word, 8),
                      __shfl_sync(0xffffffffu, word, 16), __shfl_sync(0xffffffffu, word, 24));
}
// Byte of (row j, 32-block b) in a tile's scale atoms (512-byte atoms of 4
// blocks x 128 rows: byte 16 (j mod 32) + 4 (j / 32) + (b mod 4)).
K3_DEV size_t mq_sf_off(int j, int b) { return (size_t)(b >> 2) * 512 + 16 * (j & 31) + 4 * (j >> 5) + (b & 3); }
// Byte of (row j, 32-block b) in a tile's code rows (k-step-major: k-step
// b / 8 is a block of np rows x 128 bytes, chunk b mod 8 of row j swizzled).
K3_DEV size_t mq_code_off(int j, int b, int np)
{
    return (size_t)(b >> 3) * np * 128 + (size_t)j * 128 + ((((b & 7) ^ (j & 7))) << 4);
}

// ------------------------------------------------------------------ quantiser

// rows x cols values (cols a multiple of 32) -> codes [rows][cols/2] and
// scale bytes [rows][cols/32]; one warp per 32-block.
template <typename XT>
__global__ void __launch_bounds__(256) k3_mxq_quantize(const XT *__restrict__ x, int rows, int cols,
                                                       uint8_t *__restrict__ codes, uint8_t *__restrict__ scales)
{
    const int lane = threadIdx.x & 31;
    const long nb = (long)rows * (cols / 32);
    for (long b = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nb;
         b += (long)gridDim.x * (blockDim.x >> 5)) {
        float v;
        if constexpr (sizeof(XT) == 2)
            v = __uint_as_float((uint32_t)((const uint16_t *)x)[32 * b + lane] << 16);
        else
            v = ((const float *)x)[32 * b + lane];
        uint32_t sb;
        const uint32_t word = mxq_pack(mxq_code(v, &sb), lane);
        if ((lane & 7) == 0) *(uint32_t *)(codes + 16 * b + 4 * (lane >> 3)) = word;
        if (lane == 0) scales[b] = (uint8_t)sb;
    }
}

// ---------------------------------------------------------------- planning

// Tiles of at most 128 tokens per expert (offsets from the grouping), their
// rows in the token / h arrays, and the first tile of every expert.  One CTA.
__global__ void __launch_bounds__(1024) k3_mxq_plan(const int32_t *__restrict__ offsets, int E, int max_tiles,
                                                    MqTile *tiles, int32_t *n_tiles, int32_t *tbase, int *err)
{
    __shared__ int wsum[2][32];
    __shared__ int base[2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) base[0] = base[1] = 0;
    __syncthreads();
    for (int e0 = 0; e0 < E; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        const int c = e < E ? offsets[e + 1] - offsets[e] : 0;
        const int nt = (c + MQ_TN - 1) / MQ_TN;
        const int rows = (c / MQ_TN) * MQ_TN + (((c % MQ_TN) + 15) & ~15);
        int v[2] = {nt, rows}, inc[2];
#pragma unroll
        for (int q = 0; q < 2; q++) {
            inc[q] = v[q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, inc[q], o);
                if (lane >= o) inc[q] += y;
            }
            if (lane == 31) wsum[q][warp] = inc[q];
        }
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int q = 0; q < 2; q++) {
                int s = lane < nw ? wsum[q][lane] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, s, o);
                    if (lane >= o) s += y;
                }
                if (lane < nw) wsum[q][lane] = s;
            }
        }
        __syncthreads();
        int t = base[0] + inc[0] - v[0] + (warp ? wsum[0][warp - 1] : 0);
        int r = base[1] + inc[1] - v[1] + (warp ? wsum[1][warp - 1] : 0);
        if (e < E) tbase[e] = t;
        for (int j = 0; j < nt; j++, t++) {
            const int n = min(MQ_TN, c - j * MQ_TN);
            const int np = (n + 15) & ~15;
            if (t < max_tiles) {
                MqTile tl = {};
                tl.expert = e;
                tl.pair_begin = offsets[e] + j * MQ_TN;
                tl.n = n;
                tl.np = np;
                tl.row0 = r;
                tiles[t] = tl;
            }
            r += np;
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) {
            base[0] = t;
            base[1] = r;
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

// slot[pair] = tile * 128 + row of the pair in its expert's tiles.
__global__ void __launch_bounds__(256) k3_mxq_slots(const int32_t *__restrict__ offsets, int E,
                                                    const int32_t *__restrict__ perm, int npairs,
                                                    const int32_t *__restrict__ tbase, int32_t *slot)
{
    for (int pos = blockIdx.x * blockDim.x + threadIdx.x; pos < npairs; pos += gridDim.x * blockDim.x) {
        int lo = 0, hi = E;  // the expert e with offsets[e] <= pos < offsets[e + 1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(offsets + mid) <= pos)
                lo = mid;
            else
                hi = mid;
        }
        const int idx = pos - __ldg(offsets + lo);
        slot[perm[pos]] = (tbase[lo] + idx / MQ_TN) * MQ_TN + idx % MQ_TN;
    }
}

// Each token's 32-blocks, quantised once and written into the k tiles that
// hold the token: codes into its rows of Xg, scale bytes into the tile's
// atoms in Xsf.  One warp per token at a time.
template <typename XT>
__global__ void __launch_bounds__(256) k3_mxq_xtiles(const XT *__restrict__ X, int T, int d, int k,
                                                     const int32_t *__restrict__ slot, const MqTile *__restrict__ tiles,
                                                     uint8_t *__restrict__ Xg, uint8_t *__restrict__ Xsf)
{
    const int lane = threadIdx.x & 31;
    const int nb = d / 32;
    const size_t rowb = (size_t)d / 2, sfb = (size_t)(d / 128) * 512;
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += gridDim.x * (blockDim.x >> 5)) {
        // lane i < k: the tile row of slot i
        uint8_t *xrow = nullptr, *xsf = nullptr;
        int j = 0, np = 16;
        if (lane < k) {
            const int s = slot[(size_t)t * k + lane];
            const MqTile tl = tiles[s / MQ_TN];
            j = s % MQ_TN;
            np = tl.np;
            xrow = Xg + (size_t)tl.row0 * rowb;
            xsf = Xsf + (size_t)(s / MQ_TN) * sfb;
        }
        // four blocks at a time: their scale bytes are four consecutive bytes
        // of the row's atom (one word store instead of four byte stores)
        for (int b0 = 0; b0 < nb; b0 += 4) {
            uint32_t sw = 0;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const int b = b0 + q;
                float v;
                if constexpr (sizeof(XT) == 2)
                    v = __uint_as_float((uint32_t)((const uint16_t *)X)[(size_t)t * d + 32 * b + lane] << 16);
                else
                    v = ((const float *)X)[(size_t)t * d + 32 * b + lane];
                uint32_t sb;
                const uint4 ch = mxq_chunk(mxq_pack(mxq_code(v, &sb), lane));
                sw |= sb << (8 * q);
                if (lane < k) *(uint4 *)(xrow + mq_code_off(j, b, np)) = ch;
            }
            if (lane < k) *(uint32_t *)(xsf + mq_sf_off(j, b0)) = sw;
        }
    }
}

// ----------------------------------------------------------- expert phases

struct MqArgs {
    const MqTile *tiles;
    const int32_t *n_tiles;
    const CUtensorMap *maps;  // [E][6]: gate, up, down packed planes; gate, up, down scale planes
    const uint8_t *B;         // the B rows of the phase: token codes (gate/up) or h codes (down)
    const uint8_t *Bsf;       // their scale atoms, (K / 128) x 512 bytes per tile
    uint8_t *H, *Hsf;         // gate/up output: h codes and atoms (the down phase's B)
    const int32_t *perm;      // pair of each sorted position
    const float *wsel;        // combine weight of each pair
    float *out;               // [T][d], added into
    int k, d, f;
    int *err;
};

// PH 0: gate/up + SwiGLU + h quantisation; PH 1: down + weighted combine.
template <int PH>
struct MqCfg {
    static constexpr int NA = PH == 0 ? 2 : 1;             // weight matrices per unit
    static constexpr int NS = 4;                           // pipeline stages
    static constexpr int NEPI = PH == 0 ? 8 : 4;           // epilogue warps (two per TMEM lane quadrant at PH 0)
    static constexpr int THREADS = (MQ_W_EPI + NEPI) * 32;
    static constexpr int A_BYTES = MQ_M * 128;             // one weight tile (256 of K)
    static constexpr int SC_BYTES = MQ_M * 16;             // scale box (16 k-blocks)
    static constexpr int AT_BYTES = 2 * 512;               // two A atoms per matrix per k-step
    static constexpr int B_BYTES = MQ_TN * 128;            // token / h rows of one k-step
    static constexpr int BAT_BYTES = 2 * 512;              // their two scale atoms
    static constexpr int OFF_SC = NA * A_BYTES;
    static constexpr int OFF_AT = OFF_SC + NA * SC_BYTES;
    static constexpr int OFF_B = OFF_AT + NA * AT_BYTES;   // 1024-aligned (checked below)
    static constexpr int OFF_BAT = OFF_B + B_BYTES;
    static constexpr int STAGE = ((OFF_BAT + BAT_BYTES + 1023) / 1024) * 1024;
    static constexpr int NACC = PH == 0 ? 1 : 2;           // accumulator buffers
    static constexpr int ACC_COLS = NA * MQ_TN;            // columns of one buffer
    static constexpr int TSA = NACC * ACC_COLS;            // A scale columns: stage s, matrix m at TSA + 8 (NA s + m)
    static constexpr int TSB = TSA + 8 * NA * NS;          // B scale columns: stage s at TSB + 8 s
    static constexpr int TMEM_COLS = 512;
    static constexpr int BARS = 3 * NS + 2 * 2 + 1;        // full, atoms full, empty; acc full/empty x2; fin
    static constexpr int SMEM = 1024 + NS * STAGE + 1024;
    static_assert(OFF_B % 1024 == 0, "B rows need 1024-byte alignment for the 128-byte swizzle");
    static_assert(TSB + 8 * NS <= TMEM_COLS, "TMEM layout");
    static_assert(SMEM <= 232448, "shared memory");
};

template <int PH>
__global__ void __launch_bounds__(MqCfg<PH>::THREADS, 1) k3_mxq_expert(const MqArgs a)
{
    using C = MqCfg<PH>;
    constexpr int NA = C::NA, NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(sm);
    uint64_t *bars = (uint64_t *)(sm + NS * C::STAGE);
    const int B_FULL = 0, B_AFULL = NS, B_EMPTY = 2 * NS, B_ACCF = 3 * NS, B_ACCE = B_ACCF + 2, B_FIN = B_ACCE + 2;
    uint32_t *tmem_slot = (uint32_t *)(bars + C::BARS);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    auto stage = [&](int s) { return sbase + (uint32_t)(s * C::STAGE); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = PH == 0 ? a.d : a.f;      // reduction length
    const int ROWS = PH == 0 ? a.f : a.d;   // weight rows per matrix
    const int nrb = ROWS / MQ_M;            // units per tile
    const int nks = K / 256;                // k-steps per unit
    const size_t brow = (size_t)K / 2;      // B row bytes
    const size_t bsft = (size_t)(K / 128) * 512;  // B atom bytes per tile
    const int n_units = *a.n_tiles * nrb;
    const int G = gridDim.x, cid = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; i++) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_AFULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_ACCF + i), 1);
            mbar_init(bar(B_ACCE + i), C::NEPI);
        }
        mbar_init(bar(B_FIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MQ_W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)tmem_slot;

    if (warp == MQ_W_PROD) {
        // --------------------------------------------------------- producer
        uint32_t issued[NS];
#pragma unroll
        for (int i = 0; i < NS; i++) issued[i] = 0;
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int u = cid; u < n_units && ok && !*abort_flag; u += G) {
                const int ti = u / nrb, rb = u % nrb;
                const MqTile tl = a.tiles[ti];
                const CUtensorMap *mp = a.maps + 6 * (size_t)tl.expert;
                if (tl.np < 16 || tl.np > MQ_TN || tl.np % 16) {
                    set_device_error(a.err, K3MOE_EINVAL);
                    *abort_flag = 1;
                    break;
                }
                const uint8_t *brows = a.B + (size_t)tl.row0 * brow;
                const uint8_t *bsf = a.Bsf + (size_t)ti * bsft;
                const uint32_t bbytes = (uint32_t)tl.np * 128u;
                for (int ks = 0; ks < nks; ks++, it++) {
                    const int s = it % NS;
                    if (it >= (uint32_t)NS && !tc_wait(bar(B_EMPTY + s), ((it / NS) - 1) & 1, a.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B_FULL + s),
                                          NA * (C::A_BYTES + C::SC_BYTES) + bbytes + (uint32_t)C::BAT_BYTES);
                    issued[s]++;
#pragma unroll
                    for (int m = 0; m < NA; m++) {
                        const int mat = PH == 0 ? m : 2;
                        tma_load_2d(stage(s) + (uint32_t)(m * C::A_BYTES), mp + mat, ks * 128, rb * MQ_M,
                                    bar(B_FULL + s));
                        tma_load_2d(stage(s) + (uint32_t)(C::OFF_SC + m * C::SC_BYTES), mp + 3 + mat, 16 * (ks >> 1),
                                    rb * MQ_M, bar(B_FULL + s));
                    }
                    bulk_g2s(stage(s) + (uint32_t)C::OFF_B, brows + (size_t)ks * bbytes, bbytes, bar(B_FULL + s));
                    bulk_g2s(stage(s) + (uint32_t)C::OFF_BAT, bsf + (size_t)ks * C::BAT_BYTES, C::BAT_BYTES,
                             bar(B_FULL + s));
                }
            }
            // drain: every copy issued here has landed before the CTA exits
            for (int s = 0; s < NS; s++)
                if (issued[s]) mbar_wait(bar(B_FULL + s), (issued[s] - 1) & 1, a.err);
        }
        __syncwarp();
    } else if (warp == MQ_W_PERM) {
        // ------------------------------------ scale boxes -> tcgen05.cp atoms
        // atom byte 16 r0 + 4 r1 + kb = scale of row r0 + 32 r1, k-block kb;
        // a k-step uses 8 of its box's 16 k-blocks (the half of ks mod 2)
        uint32_t it = 0;
        for (int u = cid; u < n_units && !*abort_flag; u += G) {
            for (int ks = 0; ks < nks; ks++, it++) {
                const int s = it % NS;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_FULL + s), (it / NS) & 1, a.err, abort_flag))) break;
#pragma unroll
                for (int m = 0; m < NA; m++)
#pragma unroll
                    for (int at = 0; at < 2; at++)
#pragma unroll
                        for (int r1 = 0; r1 < 4; r1++) {
                            const uint32_t box = stage(s) + (uint32_t)(C::OFF_SC + m * C::SC_BYTES);
                            uint32_t v = mq_lds32(box + (uint32_t)((lane + 32 * r1) * 16 + 8 * (ks & 1) + 4 * at));
                            v &= ~__vcmpeq4(v, 0xffffffffu);  // 255 (a dropped weight group) -> 2^-127
                            mq_sts32(stage(s) + (uint32_t)(C::OFF_AT + m * C::AT_BYTES + at * 512 + 16 * lane + 4 * r1),
                                     v);
                        }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_AFULL + s));
            }
        }
    } else if (warp == MQ_W_MMA) {
        // -------------------------------------------------------------- MMA
        uint32_t it = 0, ut = 0;
        for (int u = cid; u < n_units && !*abort_flag; u += G, ut++) {
            const MqTile tl = a.tiles[u / nrb];
            if (tl.np < 16 || tl.np > MQ_TN || tl.np % 16) {
                if (lane == 0) set_device_error(a.err, K3MOE_EINVAL);
                *abort_flag = 1;
                break;
            }
            const int buf = C::NACC == 2 ? (int)(ut & 1) : 0;
            const uint32_t uses = C::NACC == 2 ? ut / 2 : ut;  // earlier units on this buffer
            if (uses >= 1 &&
                !__all_sync(0xffffffffu, tc_wait(bar(B_ACCE + buf), (uses - 1) & 1, a.err, abort_flag)))
                break;
            tc_fence_after();
            const uint32_t tacc = tmem + (uint32_t)(buf * C::ACC_COLS);
            bool ok = true;
            for (int ks = 0; ks < nks; ks++, it++) {
                const int s = it % NS;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_AFULL + s), (it / NS) & 1, a.err, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tsa = tmem + (uint32_t)(C::TSA + 8 * NA * s), tsb = tmem + (uint32_t)(C::TSB + 8 * s);
#pragma unroll
                for (int m = 0; m < NA; m++) {
                    mq_cp_atom(tsa + 8 * m, stage(s) + (uint32_t)(C::OFF_AT + m * C::AT_BYTES));
                    mq_cp_atom(tsa + 8 * m + 4, stage(s) + (uint32_t)(C::OFF_AT + m * C::AT_BYTES + 512));
                }
                mq_cp_atom(tsb, stage(s) + (uint32_t)C::OFF_BAT);
                mq_cp_atom(tsb + 4, stage(s) + (uint32_t)(C::OFF_BAT + 512));
                const uint32_t blo = sw128_lo(stage(s) + (uint32_t)C::OFF_B);
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {  // K = 64 per MMA
                    const uint32_t idesc = mq_idesc(tl.np, 2u * (q4 & 1), 2u * (q4 & 1));
#pragma unroll
                    for (int m = 0; m < NA; m++)
                        mq_mma(tacc + (uint32_t)(m * MQ_TN), sw128_lo(stage(s) + (uint32_t)(m * C::A_BYTES)) + 2u * q4,
                               blo + 2u * q4, idesc, tsa + 8 * m + 4 * (q4 >> 1), tsb + 4 * (q4 >> 1),
                               (ks == 0 && q4 == 0) ? 0u : 1u);
                }
                mma_commit(bar(B_EMPTY + s));
            }
            if (!ok) break;
            mma_commit(bar(B_ACCF + buf));
        }
        // every MMA and copy issued above has completed before TMEM is freed
        mma_commit(bar(B_FIN));
        mbar_wait(bar(B_FIN), 0, a.err);
        __syncwarp();
    } else if (warp >= MQ_W_EPI) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant: weight rows 32 q .. 32 q + 31 of the unit
        const int half = (warp - MQ_W_EPI) >> 2;  // PH 0: the two warps of a quadrant take alternate chunks
        uint32_t ut = 0;
        for (int u = cid; u < n_units && !*abort_flag; u += G, ut++) {
            const int ti = u / nrb, rb = u % nrb;
            const MqTile tl = a.tiles[ti];
            const int buf = C::NACC == 2 ? (int)(ut & 1) : 0;
            const uint32_t uses = C::NACC == 2 ? ut / 2 : ut;
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_ACCF + buf), uses & 1, a.err, abort_flag))) break;
            tc_fence_after();
            const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * C::ACC_COLS);
            if (PH == 0) {
                // h = silu(g) * u for rows 128 rb + 32 q + lane of f (one 32-block of
                // the down product's K) and 8 tokens at a time, quantised and
                // written as chunk 4 (rb mod 2) + q of k-step rb / 2 of each token's
                // h row; its scale byte into atom rb
                uint8_t *hrows = a.H + (size_t)tl.row0 * (a.f / 2);
                uint8_t *hsf = a.Hsf + (size_t)ti * (size_t)(a.f / 128) * 512;
                const int b = 4 * rb + q;  // 32-block of f
                bool released = false;
                for (int j0 = 8 * half; j0 < tl.n; j0 += 16) {
                    float g[8], v[8];
                    tmem_ld8(tacc + (uint32_t)j0, g);
                    tmem_ld8(tacc + (uint32_t)(MQ_TN + j0), v);
                    tmem_wait_ld();
                    if (j0 + 16 >= tl.n) {
                        // this warp's columns are read: once every epilogue warp
                        // has done so, the next unit's MMAs may start
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_ACCE + buf));
                        released = true;
                    }
                    // eight tokens at once: their block maxima, this row's eight
                    // codes as one word (nibble i = token j0 + i), then a nibble
                    // transpose leaves word lane / 8 of token j0 + lane % 8's
                    // 16-byte chunk in each lane
                    uint32_t ab[8], mb[8], w = 0u, myscale = 0u;
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float h = silu(g[i]) * v[i];
                        ab[i] = __float_as_uint(h);
                        mb[i] = __reduce_max_sync(0xffffffffu, ab[i] & 0x7fffffffu);
                    }
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        uint32_t e;
                        const uint32_t c = mxq_rule(ab[i] & 0x7fffffffu, ab[i] >> 31, mb[i], e);
                        w |= c << (4 * i);
                        if (lane == i) myscale = e;
                    }
                    w = nib_transpose8(w, lane);
                    const int j = j0 + (lane & 7);
                    if (j < tl.n) {
                        *(uint32_t *)(hrows + mq_code_off(j, b, tl.np) + 4 * (lane >> 3)) = w;
                        if (lane < 8) hsf[mq_sf_off(j, b)] = (uint8_t)myscale;
                    }
                }
                if (!released) {  // no chunk of this unit fell to this warp
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_ACCE + buf));
                }
            } else {
                // lane l of group g (rows 8 g .. 8 g + 7 of this warp's 32) takes
                // token j0 + (l mod 8) of the eight and adds its eight rows with
                // two vector reductions
                for (int j0 = 0; j0 < tl.n; j0 += 8) {
                    float y[8];
                    tmem_ld8(tacc + (uint32_t)j0, y);
                    tmem_wait_ld();
                    mq_transpose8(y, lane);
                    const int j = j0 + (lane & 7);
                    if (j < tl.n) {
                        const int pair = a.perm[tl.pair_begin + j];
                        const float w = a.wsel[pair];
                        float *o = a.out + (size_t)(pair / a.k) * a.d + rb * MQ_M + q * 32 + (lane & ~7);
                        mq_red_v4(o, w * y[0], w * y[1], w * y[2], w * y[3]);
                        mq_red_v4(o + 4, w * y[4], w * y[5], w * y[6], w * y[7]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_ACCE + buf));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MQ_W_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
    }
}

// ------------------------------------------------------- down (resident h)

// Down products, units (tile, 128 rows of d) taken group by group (8 row
// blocks of d per group, every group split evenly over the CTAs, tile-major
// within it): the weighted reductions of all CTAs then land in the same
// 8 x 128 columns of out at any time, which stay in L2.  A tile's h codes
// (np x f/2 bytes) and scale atoms are copied into shared memory once per
// run of its row blocks and stay there while the down weight tiles stream
// through a ring of stages.
constexpr int MD_NS = 6;                        // weight stages
constexpr int MD_RG = 8;                        // row blocks of d per group (locality of the reductions)
constexpr int MD_STAGE = MQ_M * 128 + MQ_M * 16 + 1024;  // A tile, scale box, A atoms
constexpr int MD_HMAX = MQ_TN * 768;            // h codes of a tile at most (f <= 1536)
constexpr int MD_HSF = 12 * 512;                // its scale atoms (f / 128 <= 12)
constexpr int MD_OFF_H = MD_NS * MD_STAGE;      // 1024-aligned: the stage is
constexpr int MD_SMEM = 1024 + MD_OFF_H + MD_HMAX + MD_HSF + 1024;
static_assert(MD_STAGE % 1024 == 0 && MD_SMEM <= 232448, "down smem");
constexpr int MD_TACC = 0, MD_TSA = 2 * MQ_TN, MD_TSB = MD_TSA + 8 * MD_NS;  // + 2 x 48 B-scale columns
static_assert(MD_TSB + 2 * 48 <= 512, "down TMEM");

__global__ void __launch_bounds__(MQ_THREADS, 1) k3_mxq_down(const MqArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_addr(sm);
    uint64_t *bars = (uint64_t *)(sm + MD_OFF_H + MD_HMAX + MD_HSF);
    const int B_FULL = 0, B_AFULL = MD_NS, B_EMPTY = 2 * MD_NS, B_ACCF = 3 * MD_NS, B_ACCE = B_ACCF + 2,
              B_HFULL = B_ACCE + 2, B_HFREE = B_HFULL + 1, B_FIN = B_HFREE + 1, NB = B_FIN + 1;
    uint32_t *tmem_slot = (uint32_t *)(bars + NB);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    auto stage = [&](int s) { return sbase + (uint32_t)(s * MD_STAGE); };
    const uint32_t hbuf = sbase + (uint32_t)MD_OFF_H, hsfbuf = hbuf + (uint32_t)MD_HMAX;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrb = a.d / MQ_M, nks = a.f / 256;
    const int n_tiles = *a.n_tiles;
    const int ngrp = (nrb + MD_RG - 1) / MD_RG;
    const long G = gridDim.x;
    // This CTA's units, group after group: in group g (row blocks MD_RG g ..
    // MD_RG g + rg - 1) the n_tiles x rg units (tile-major) are split evenly
    // over the CTAs, so that at any time the CTAs add into the same rg x 128
    // columns of out (a few MB, kept in L2).  seq(i) gives the i-th unit of
    // this CTA as (tile, row block).
    auto grp_lo = [&](int g) {
        const long ug = (long)n_tiles * min(MD_RG, nrb - MD_RG * g);
        return ug * blockIdx.x / G;
    };
    auto grp_hi = [&](int g) {
        const long ug = (long)n_tiles * min(MD_RG, nrb - MD_RG * g);
        return ug * (blockIdx.x + 1) / G;
    };
    long my_units = 0;
    for (int g = 0; g < ngrp; g++) my_units += grp_hi(g) - grp_lo(g);
    const long ulo = 0, uhi = my_units;
    // cursor over the sequence (each role keeps its own)
    struct Cursor {
        int g;
        long v, hi;
    };
    auto cur_init = [&]() {
        Cursor c{0, grp_lo(0), grp_hi(0)};
        while (c.v >= c.hi && c.g + 1 < ngrp) {
            c.g++;
            c.v = grp_lo(c.g);
            c.hi = grp_hi(c.g);
        }
        return c;
    };
    auto cur_next = [&](Cursor &c) {
        c.v++;
        while (c.v >= c.hi && c.g + 1 < ngrp) {
            c.g++;
            c.v = grp_lo(c.g);
            c.hi = grp_hi(c.g);
        }
    };
    auto cur_tile = [&](const Cursor &c) { return (int)(c.v / min(MD_RG, nrb - MD_RG * c.g)); };
    auto cur_rb = [&](const Cursor &c) { return MD_RG * c.g + (int)(c.v % min(MD_RG, nrb - MD_RG * c.g)); };
    const uint32_t hrow = (uint32_t)a.f / 2, hsfb = (uint32_t)(a.f / 128) * 512;

    if (threadIdx.x == 0) {
        for (int i = 0; i < MD_NS; i++) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_AFULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(bar(B_ACCF + i), 1);
            mbar_init(bar(B_ACCE + i), 4);
        }
        mbar_init(bar(B_HFULL), 1);
        mbar_init(bar(B_HFREE), 1);
        mbar_init(bar(B_FIN), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MQ_W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)tmem_slot;

    if (warp == MQ_W_PROD) {
        // ------------------------------------- weight tiles; h once per run
        uint32_t issued[MD_NS];
#pragma unroll
        for (int i = 0; i < MD_NS; i++) issued[i] = 0;
        uint32_t runs = 0;
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            int cur = -1;
            Cursor cu = cur_init();
            for (long u = ulo; u < uhi && ok && !*abort_flag; u++, cur_next(cu)) {
                const int ti = cur_tile(cu), rb = cur_rb(cu);
                const MqTile tl = a.tiles[ti];
                if (tl.np < 16 || tl.np > MQ_TN || tl.np % 16 || a.f > 1536) {
                    set_device_error(a.err, K3MOE_EINVAL);
                    *abort_flag = 1;
                    break;
                }
                if (ti != cur) {
                    // the previous run's MMAs are done with the h buffer
                    if (runs >= 1 && !tc_wait(bar(B_HFREE), (runs - 1) & 1, a.err, abort_flag)) break;
                    cur = ti;
                    const uint32_t hb = (uint32_t)tl.np * hrow;
                    mbar_arrive_expect_tx(bar(B_HFULL), hb + hsfb);
                    for (uint32_t o = 0; o < hb; o += 32768)
                        bulk_g2s(hbuf + o, a.B + (size_t)tl.row0 * hrow + o, min(32768u, hb - o), bar(B_HFULL));
                    bulk_g2s(hsfbuf, a.Bsf + (size_t)ti * hsfb, hsfb, bar(B_HFULL));
                    runs++;
                }
                const CUtensorMap *mp = a.maps + 6 * (size_t)tl.expert;
                for (int ks = 0; ks < nks; ks++, it++) {
                    const int s = it % MD_NS;
                    if (it >= (uint32_t)MD_NS &&
                        !tc_wait(bar(B_EMPTY + s), ((it / MD_NS) - 1) & 1, a.err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B_FULL + s), MQ_M * 128 + MQ_M * 16);
                    issued[s]++;
                    tma_load_2d(stage(s), mp + 2, ks * 128, rb * MQ_M, bar(B_FULL + s));
                    tma_load_2d(stage(s) + MQ_M * 128, mp + 5, 16 * (ks >> 1), rb * MQ_M, bar(B_FULL + s));
                }
            }
            for (int s = 0; s < MD_NS; s++)
                if (issued[s]) mbar_wait(bar(B_FULL + s), (issued[s] - 1) & 1, a.err);
            if (runs) mbar_wait(bar(B_HFULL), (runs - 1) & 1, a.err);
        }
        __syncwarp();
    } else if (warp == MQ_W_PERM) {
        // ------------------------------------ scale boxes -> tcgen05.cp atoms
        uint32_t it = 0;
        for (long u = ulo; u < uhi && !*abort_flag; u++) {
            for (int ks = 0; ks < nks; ks++, it++) {
                const int s = it % MD_NS;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_FULL + s), (it / MD_NS) & 1, a.err, abort_flag))) break;
#pragma unroll
                for (int at = 0; at < 2; at++)
#pragma unroll
                    for (int r1 = 0; r1 < 4; r1++) {
                        uint32_t v = mq_lds32(stage(s) + MQ_M * 128 + (uint32_t)((lane + 32 * r1) * 16 + 8 * (ks & 1) + 4 * at));
                        v &= ~__vcmpeq4(v, 0xffffffffu);  // 255 (a dropped weight group) -> 2^-127
                        mq_sts32(stage(s) + MQ_M * 144 + (uint32_t)(at * 512 + 16 * lane + 4 * r1), v);
                    }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_AFULL + s));
            }
            if (*abort_flag) break;
        }
    } else if (warp == MQ_W_MMA) {
        // -------------------------------------------------------------- MMA
        uint32_t it = 0, ut = 0, runs = 0;
        int cur = -1;
        bool ok = true;
        Cursor cu = cur_init();
        for (long u = ulo; u < uhi && ok && !*abort_flag; u++, ut++, cur_next(cu)) {
            const int ti = cur_tile(cu);
            const MqTile tl = a.tiles[ti];
            if (ti != cur) {
                if (runs >= 1) mma_commit(bar(B_HFREE));  // the previous run's MMAs release the h buffer
                cur = ti;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_HFULL), runs & 1, a.err, abort_flag))) break;
                tc_fence_after();
                const uint32_t tsb = tmem + (uint32_t)(MD_TSB + 48 * (runs & 1));
                for (int at = 0; at < a.f / 128; at++) mq_cp_atom(tsb + 4 * at, hsfbuf + (uint32_t)(512 * at));
                runs++;
            }
            const int buf = (int)(ut & 1);
            if (ut >= 2 && !__all_sync(0xffffffffu, tc_wait(bar(B_ACCE + buf), ((ut / 2) - 1) & 1, a.err, abort_flag)))
                break;
            tc_fence_after();
            const uint32_t tacc = tmem + (uint32_t)(MD_TACC + buf * MQ_TN);
            const uint32_t tsb = tmem + (uint32_t)(MD_TSB + 48 * ((runs - 1) & 1));
            for (int ks = 0; ks < nks; ks++, it++) {
                const int s = it % MD_NS;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_AFULL + s), (it / MD_NS) & 1, a.err, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tsa = tmem + (uint32_t)(MD_TSA + 8 * s);
                mq_cp_atom(tsa, stage(s) + MQ_M * 144);
                mq_cp_atom(tsa + 4, stage(s) + MQ_M * 144 + 512);
                const uint32_t blo = sw128_lo(hbuf + (uint32_t)(ks * tl.np * 128));
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++)
                    mq_mma(tacc, sw128_lo(stage(s)) + 2u * q4, blo + 2u * q4, mq_idesc(tl.np, 2u * (q4 & 1), 2u * (q4 & 1)),
                           tsa + 4 * (q4 >> 1), tsb + 8 * ks + 4 * (q4 >> 1), (ks == 0 && q4 == 0) ? 0u : 1u);
                mma_commit(bar(B_EMPTY + s));
            }
            if (!ok) break;
            mma_commit(bar(B_ACCF + buf));
        }
        mma_commit(bar(B_FIN));
        mbar_wait(bar(B_FIN), 0, a.err);
        __syncwarp();
    } else if (warp >= MQ_W_EPI) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        uint32_t ut = 0;
        // lane l of group g (rows 8 g .. 8 g + 7 of this warp's 32) takes
        // tokens 8 i + (l mod 8) of the tile and adds their eight rows with
        // two vector reductions.  Their output rows and combine weights are
        // read once per run of a tile's row blocks (all loads in flight
        // together), not once per token group of every unit.
        constexpr int NJ = MQ_TN / 8;
        int cur = -1, n = 0;
        size_t orow[NJ];
        float wv[NJ];
        Cursor cu = cur_init();
        for (long u = ulo; u < uhi && !*abort_flag; u++, ut++, cur_next(cu)) {
            const int ti = cur_tile(cu), rb = cur_rb(cu);
            if (ti != cur) {
                cur = ti;
                const MqTile tl = a.tiles[ti];
                n = tl.n;
                int pr[NJ];
#pragma unroll
                for (int i = 0; i < NJ; i++) {
                    const int j = 8 * i + (lane & 7);
                    pr[i] = j < n ? a.perm[tl.pair_begin + j] : 0;
                }
#pragma unroll
                for (int i = 0; i < NJ; i++) {
                    const int j = 8 * i + (lane & 7);
                    wv[i] = j < n ? a.wsel[pr[i]] : 0.f;
                    orow[i] = (size_t)(pr[i] / a.k) * a.d;
                }
            }
            const int buf = (int)(ut & 1);
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_ACCF + buf), (ut / 2) & 1, a.err, abort_flag))) break;
            tc_fence_after();
            const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(MD_TACC + buf * MQ_TN);
            const size_t col = (size_t)rb * MQ_M + q * 32 + (lane & ~7);
#pragma unroll
            for (int i = 0; i < NJ; i++) {
                if (8 * i < n) {
                    float y[8];
                    tmem_ld8(tacc + (uint32_t)(8 * i), y);
                    tmem_wait_ld();
                    mq_transpose8(y, lane);
                    if (8 * i + (lane & 7) < n) {
                        float *o = a.out + orow[i] + col;
                        const float w = wv[i];
                        mq_red_v4(o, w * y[0], w * y[1], w * y[2], w * y[3]);
                        mq_red_v4(o + 4, w * y[4], w * y[5], w * y[6], w * y[7]);
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
    if (warp == MQ_W_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

// --------------------------------------------------------------- launchers

int num_sms();

// Shapes the MXFP4-activation path takes: whole 256-long k-steps and 128-row
// weight tiles on both products (and E8M0 16-byte scale boxes: K a multiple
// of 512).
bool mxq_supported(int E, int k, int d, int f)
{
    return E >= 1 && k >= 1 && k <= 16 && d % 512 == 0 && f % 512 == 0 && d <= 16384 && f <= 16384;
}
int mxq_max_tiles(int npairs, int E) { return (npairs + MQ_TN - 1) / MQ_TN + E; }
size_t mxq_max_rows(int npairs, int E) { return (size_t)npairs + 15 * (size_t)E; }
size_t mxq_tile_bytes() { return sizeof(MqTile); }

// Quantises rows x cols values (bf16 or fp32) by the OCP MX rule.
int launch_mx_quantize(const void *x, int xdt, int rows, int cols, uint8_t *codes, uint8_t *scales, cudaStream_t s)
{
    const long nb = (long)rows * (cols / 32);
    const int grid = (int)std::min<long>((nb + 7) / 8, 16L * num_sms());
    if (xdt == K3MOE_BF16)
        k3_mxq_quantize<uint16_t><<<grid, 256, 0, s>>>((const uint16_t *)x, rows, cols, codes, scales);
    else
        k3_mxq_quantize<float><<<grid, 256, 0, s>>>((const float *)x, rows, cols, codes, scales);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

template <int PH>
static int launch_mxq_phase(const MqArgs &a, cudaStream_t s)
{
    using C = MqCfg<PH>;
    if (ensure_smem((const void *)k3_mxq_expert<PH>, C::SMEM) != K3MOE_OK) return K3MOE_ECUDA;
    k3_mxq_expert<PH><<<num_sms(), C::THREADS, C::SMEM, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

// The gate/up half of a grouped batch with MXFP4 activations: tile plan,
// token tiles, gate/up + SwiGLU with h quantised into Hg / Hsf.  offsets /
// perm from the grouping; maps: the layer's six tensor maps per expert.
int launch_mxq_gateup(const void *X, int xdt, int T, int k, int E, int d, int f, const void *maps,
                      const int32_t *offsets, const int32_t *perm, void *tiles, int32_t *n_tiles, int32_t *tbase,
                      int32_t *slot, int max_tiles, uint8_t *Xg, uint8_t *Xsf, uint8_t *Hg, uint8_t *Hsf, int *err,
                      cudaStream_t s)
{
    const int npairs = T * k;
    k3_mxq_plan<<<1, 1024, 0, s>>>(offsets, E, max_tiles, (MqTile *)tiles, n_tiles, tbase, err);
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    k3_mxq_slots<<<std::max(1, std::min((npairs + 255) / 256, 4 * num_sms())), 256, 0, s>>>(offsets, E, perm, npairs,
                                                                                           tbase, slot);
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    const int xg = std::max(1, std::min((T + 7) / 8, 8 * num_sms()));
    if (xdt == K3MOE_BF16)
        k3_mxq_xtiles<uint16_t><<<xg, 256, 0, s>>>((const uint16_t *)X, T, d, k, slot, (const MqTile *)tiles, Xg, Xsf);
    else
        k3_mxq_xtiles<float><<<xg, 256, 0, s>>>((const float *)X, T, d, k, slot, (const MqTile *)tiles, Xg, Xsf);
    if (cudaGetLastError() != cudaSuccess) return K3MOE_ECUDA;
    MqArgs a = {};
    a.tiles = (const MqTile *)tiles;
    a.n_tiles = n_tiles;
    a.maps = (const CUtensorMap *)maps;
    a.perm = perm;
    a.k = k;
    a.d = d;
    a.f = f;
    a.err = err;
    a.B = Xg;
    a.Bsf = Xsf;
    a.H = Hg;
    a.Hsf = Hsf;
    return launch_mxq_phase<0>(a, s);
}

// The down half: down products of the same tiles, w * y added into out
// (zeroed first).
int launch_mxq_down(int T, int k, int d, int f, const void *maps, const int32_t *perm, const float *wsel,
                    const void *tiles, const int32_t *n_tiles, const uint8_t *Hg, const uint8_t *Hsf, float *out,
                    int *err, cudaStream_t s)
{
    MqArgs a = {};
    a.tiles = (const MqTile *)tiles;
    a.n_tiles = n_tiles;
    a.maps = (const CUtensorMap *)maps;
    a.perm = perm;
    a.wsel = wsel;
    a.k = k;
    a.d = d;
    a.f = f;
    a.err = err;
    a.B = Hg;
    a.Bsf = Hsf;
    a.out = out;
    if (cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * d, s) != cudaSuccess) return K3MOE_ECUDA;
    if (f > 1536) return launch_mxq_phase<1>(a, s);
    if (ensure_smem((const void *)k3_mxq_down, MD_SMEM) != K3MOE_OK) return K3MOE_ECUDA;
    k3_mxq_down<<<num_sms(), MQ_THREADS, MD_SMEM, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

}  // namespace k3
