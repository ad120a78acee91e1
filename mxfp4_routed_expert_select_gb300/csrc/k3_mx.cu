// k3_mx.cu -- batch-1 expert products on the block-scaled tensor cores.
//
// The pages' expert weights are E2M1 codes with one E8M0 scale per 32
// ("kimi-k3-in-c" explainer, "Reduction one"), which is exactly the operand
// format of tcgen05.mma kind::mxf4 (block_scale, scale_vec::2X): packed
// E2M1 A and B in shared memory, one E8M0 scale per row and 32 of K in TMEM.
// So the packed planes go from HBM to the tensor core by TMA with no decode
// at all, and the fp32 activations become the B operand as a sum of E2M1
// pieces:
//
//   v = sum_p q_p * 2^(s_p)      per 32-block of v, p = 0..15
//
// where, E being the biased exponent of the block's largest magnitude, q_p
// is the p-th base-4 digit (from the top) of the 32-bit fixed-point
// magnitude |v| * 2^(158 - E), as an E2M1 value 0, .5, 1 or 1.5 with the sign
// of v, and s_p = E - 127 - 2p (k3_mx.cuh, mx_encode_block).  Values down to
// 2^-8 of the block's scale are represented exactly, smaller ones to 2^-32 of
// it.  The 16 pieces are the 16 columns of one M = 128, N = 16 MMA; the
// epilogue adds the columns, smallest first.
//
// Per token, one launch of one CTA per SM, all resident at once:
//   router   logits of this CTA's block of router rows, a grid barrier, then
//            every CTA selects the top k itself (k rounds of a warp maximum
//            per warp, then a rank over the warps' candidates) and the pieces of x
//            are copied in: a B image [K/256][16 rows][128 bytes], 128-byte
//            swizzled, plus E8M0 scale atoms [K/128][512 bytes] in the layout
//            tcgen05.cp copies to TMEM
//   phase 0  gate and up rows of the k experts (tiles of 128 rows, K = d):
//            g, u -> h = silu(g) * u -> the pieces of h per expert (B images
//            of phase 1)
//   phase 1  down rows (tiles of 128 rows, K = f): y_j -> out = sum_j w_j y_j
// Both phases split the k * rows/128 tiles' K steps evenly over the CTAs (a
// tile may be split between CTAs).  The CTA holding a split tile's first
// units (at the end of its range) finishes the tile: it waits for the other
// segments' partial sums, published early in the ranges of the CTAs after
// it, while its own MMAs still run, and adds them in a fixed order, so the
// result does not depend on timing.  The launch is a programmatic dependent
// of the previous kernel on the stream: the router rows are requested before
// that kernel has finished, everything else after it.
//
// A weight group whose scale byte is 255 is dropped, as on the other paths:
// its scale becomes 0 (2^-127), so it adds at most 6 * 2^-127 * sum |v| of
// its block, far below the fp32 resolution of any nonzero output.
//
// Each phase runs as two waves, the first k * 3/4 expert slots and then the
// rest (gate/up A, gate/up B, down A, down B), so that down A starts on an h
// that was completed while gate/up B streamed, and h of B is completed while
// down A streams: the copy engines never wait for an epilogue.
//
// CTA: 12 warps.  warp 0 TMA producer (weight tiles 128 rows x 128 bytes,
// scale boxes 128 rows x 16 bytes), warp 1 MMA issuer and TMEM owner, warp
// 2 turns scale boxes into tcgen05.cp atoms, warp 3 loads phase 1's h
// pieces, warps 4-7 the phase-0 epilogue and warps 8-11 the phase-1
// epilogue (TMEM lane quadrants 0-3 each), so that down products are taken
// out of TMEM while the last gate/up tiles are still being finished.  Every
// wait is bounded; a timeout sets the device error word and the CTA drains
// and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "k3_mx.cuh"
#include "k3_tcgen05.cuh"

namespace k3 {

constexpr int MX_M = 128;       // weight rows per tile
constexpr int MX_UK = 256;      // K per unit: 128 packed bytes per row, 4 MMAs
constexpr int MX_THREADS = 384;
constexpr int MX_W_PROD = 0, MX_W_MMA = 1, MX_W_PERM = 2, MX_W_BLD = 3, MX_W_EPI = 4, MX_W_EPI1 = 8;
constexpr int MX_TMEM_COLS = 512;
constexpr int MX_ROUTER_ROWS = 8;  // router rows per CTA at most (E <= 8 x the SM count)

// Instruction descriptor of kind::mxf4 block_scale: E2M1 A and B (format 1,
// bits 7-9 and 10-12), K-major, N = 16 (bits 17-22: N >> 3), UE8M0 scales
// (bit 23), M = 128 (bits 24-28: M >> 4), the byte of the A and B scale
// words that holds this MMA's first scale (bits 29-30 and 4-5).
K3_DEV uint32_t mx_idesc(uint32_t ida, uint32_t idb)
{
    return (idb << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MX_N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(MX_M >> 4) << 24) | (ida << 29);
}
// One MMA, issued by the elected lane of a converged warp.
K3_DEV void mx_mma(uint32_t td, uint32_t alo, uint32_t blo, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                   uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "mov.b64 da, {%1, %7};\n\tmov.b64 db, {%2, %7};\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], da, db, %3, [%5], [%6], p;\n\t}"
                 ::"r"(td), "r"(alo), "r"(blo), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb), "r"(SW128_HI)
                 : "memory");
}
// Copies one 512-byte scale atom (32 rows x 16 bytes, no swizzle) from shared
// memory to TMEM columns taddr .. taddr+3 of lanes 0-31, repeated in the
// other three lane quadrants.
K3_DEV void mx_cp_atom(uint32_t taddr, uint32_t saddr)
{
    const uint32_t lo = ((saddr & 0x3FFFFu) >> 4) | (1u << 16), hi = (128u >> 4) | (1u << 14);
    asm volatile("{\n\t.reg .pred e;\n\t.reg .b64 d;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "mov.b64 d, {%1, %2};\n\t@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], d;\n\t}" ::"r"(taddr),
                 "r"(lo), "r"(hi)
                 : "memory");
}
K3_DEV uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
K3_DEV void sts32(uint32_t a, uint32_t v) { asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory"); }
// Named barrier of the four epilogue warps.  The non-aligned form: a lane
// that arrives after the others of its warp (the leader after its ticket)
// is counted as itself, not as another arrival of the whole warp.
// CTA-wide barrier in its non-aligned form: every thread is counted as
// itself, so a warp whose lanes come from different role code (lane 0 of the
// producer after its loop, the epilogue leader after its counts) cannot be
// counted twice and let the barrier open before another warp arrives.
K3_DEV void cta_sync_threads() { asm volatile("barrier.sync 0;" ::: "memory"); }
K3_DEV void red_add_f32(float *p, float v) { asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory"); }
// Named barrier of one phase's four epilogue warps (2: phase 0, 3: phase 1;
// the two groups run at the same time).
template <int PH>
K3_DEV void mx_bar_epi()
{
    if (PH == 0) asm volatile("barrier.sync 2, 128;" ::: "memory");
    else asm volatile("barrier.sync 3, 128;" ::: "memory");
}
K3_DEV unsigned ticket_add(unsigned *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

struct MxArgs {
    const CUtensorMap *maps;  // [E][6]: gate, up, down packed planes; gate, up, down scale planes
    const uint8_t *bimg;      // phase 0: x pieces [d/256][16][128]; phase 1: h pieces, per slot j
    const uint8_t *bsf;       // phase 0: x scale atoms [d/128][512]; phase 1: per slot j
    uint8_t *himg, *hsf;      // phase 0 output: h pieces per slot j (f * 8 and f / 128 * 512 bytes)
    float *part;              // split-tile partials of phase 0 [tiles][units per tile][128][2]
    float *out;               // phase 1: [d], added into
    unsigned *cnt;            // phase 0: [tiles] tickets; phase 1: [d / 128] row-tile tickets
    int k, d, f;
    int *err;
};

// A stage holds two 128-row x 128-byte A tiles: phase 0 the gate and the up
// tile of one 256-long K step (two accumulators), phase 1 two consecutive
// 256-long K steps of the down rows (one accumulator, a 512-long unit).
// Scale boxes (128 rows x 16 bytes = 16 k-blocks): phase 0 one per matrix,
// of which a unit uses half; phase 1 one, all of it.
template <int PH>
struct MxCfg {
    static constexpr int NMAT = 2;                       // A tiles per stage
    static constexpr int NOUT = PH == 0 ? 2 : 1;         // accumulators
    static constexpr int NSC = PH == 0 ? 2 : 1;          // scale boxes per stage
    static constexpr int UK = PH == 0 ? 256 : 512;       // K per unit
    static constexpr int A_BYTES = MX_M * 128;           // one A tile
    static constexpr int SC_BYTES = MX_M * 16;           // scale box
    static constexpr int AT_BYTES = 2 * 512;             // two atoms per A tile
    static constexpr int STAGE = NMAT * (A_BYTES + AT_BYTES) + NSC * SC_BYTES;
    static constexpr int NS = PH == 0 ? 4 : 5;
    // TMEM columns: accumulators from TACC, A scale slots from TSA, B scales
    // from TSB.  Phase 1 uses the columns of phase 0's B scales (free once
    // phase 0's MMAs are done), so its MMAs can start while the phase-0
    // epilogue still reads phase 0's accumulators (columns 0-63).
    static constexpr int TACC = PH == 0 ? 0 : 128;
    static constexpr int TSA = PH == 0 ? 64 : 160, TSB = PH == 0 ? 128 : 240;
    static constexpr int TMEM_COLS = 512;
    static_assert(TACC + NOUT * 2 * MX_N <= TSA && NS * NMAT * 8 <= TSB - TSA, "TMEM layout");
};

// Shared memory of one phase: [stages][B images][scale atom staging (phase 1)].
// The phases overlap; the barriers of both follow the larger layout.
template <int PH>
static size_t mx_layout_bytes(int K)
{
    using C = MxCfg<PH>;
    const size_t b = PH == 0 ? (size_t)K * 8 : 2 * (size_t)K * 8;
    const size_t sf = PH == 0 ? 0 : 2 * (size_t)(K / 128) * 512;
    return (size_t)C::NS * C::STAGE + b + sf;
}
static size_t mx_bar_off(int d, int f) { return std::max(mx_layout_bytes<0>(d), mx_layout_bytes<1>(f)); }
static size_t mx_smem(int d, int f) { return 1024 + mx_bar_off(d, f) + 1024; }

// Barriers of one phase: full, atoms-full, empty per stage; accumulator
// full / empty per TMEM buffer; B image loaded per B buffer (phase 1: two
// buffers, used by the experts of a CTA's ranges in turn); B scales in TMEM;
// all MMAs done; B buffer free (phase 1: the MMAs reading it are done).
template <int PH>
struct MxBars {
    static constexpr int NS = MxCfg<PH>::NS;
    static constexpr int FULL = 0, AFULL = NS, EMPTY = 2 * NS, ACCF = 3 * NS, ACCE = ACCF + 2, BLOAD = ACCE + 2,
                         BSCL = BLOAD + 2, FIN = BSCL + 1, BFREE = FIN + 1, N = BFREE + 2;
};
template <int PH>
K3_DEV void mx_init_bars(uint64_t *bars)
{
    using Bs = MxBars<PH>;
    for (int i = 0; i < Bs::NS; i++) {
        mbar_init(smem_addr(bars + Bs::FULL + i), 1);
        mbar_init(smem_addr(bars + Bs::AFULL + i), 1);
        mbar_init(smem_addr(bars + Bs::EMPTY + i), 1);
    }
    for (int i = 0; i < 2; i++) {
        mbar_init(smem_addr(bars + Bs::ACCF + i), 1);
        mbar_init(smem_addr(bars + Bs::ACCE + i), 4);
        mbar_init(smem_addr(bars + Bs::BLOAD + i), 1);
        mbar_init(smem_addr(bars + Bs::BFREE + i), 1);
    }
    mbar_init(smem_addr(bars + Bs::BSCL), 1);
    mbar_init(smem_addr(bars + Bs::FIN), 1);
}

// Before the first fill of phase-1 stage s (bytes [s, s + 1) x STAGE of phase
// 1): the phase-0 stages under it are read for the last time (the final phase
// of their `empty` barriers, issued[q] fills ago), and if it reaches past
// phase 0's stages, into the B image of x, all of phase 0's MMAs are done
// (fin).  Only the producer thread calls it, with its own phase-0 counts.
K3_DEV bool mx_phase1_slot_free(int s, const uint64_t *bars0, const uint32_t *issued0, uint32_t fin, int *err,
                                volatile int *abort_flag)
{
    using C0 = MxCfg<0>;
    using C1 = MxCfg<1>;
    const int lo = s * C1::STAGE, hi = (s + 1) * C1::STAGE;  // bytes of phase-1 stage s
    if (hi > C0::NS * C0::STAGE) return tc_wait(fin, 0, err, abort_flag);
    for (int q = lo / C0::STAGE; q <= (hi - 1) / C0::STAGE; q++) {
        if (issued0[q] == 0u) return tc_wait(fin, 0, err, abort_flag);  // never filled: be safe
        if (!tc_wait(smem_addr(bars0 + MxBars<0>::EMPTY + q), (issued0[q] - 1u) & 1u, err, abort_flag)) return false;
    }
    return true;
}

// Bounded wait until *p >= target (acquire); false after the time limit.
K3_DEV bool mx_wait_count(const unsigned *p, unsigned target, int *err)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        __nanosleep(64);
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            set_device_error(err, K3MOE_ETIMEOUT);
            return false;
        }
    }
}

// A wave of one phase: the units [uw0, uw0 + Uw) (the tiles of a run of
// expert slots), spread over the CTAs like a whole phase.  A phase runs as
// one or two waves; first / last mark its first and last wave.
struct MxWave {
    int uw0, Uw;  // units fit in 32 bits (at most 16 x 12 x 28 per wave)
    bool first, last;
};
// What one thread's role has done in a phase so far (ring stages, finished
// accumulators, phase 1's B buffers), carried from one wave to the next so
// that every barrier's parity follows on.
template <int PH>
struct MxState {
    uint32_t it = 0, sg = 0;
    int nexp = 0, cur_j = -1;
    int pre = 0;  // producer: units of the wave already issued by mx_preissue
    uint32_t issued[MxCfg<PH>::NS] = {};
};

// The copies of one unit into ring stage s: phase 0 the gate and up tiles
// (K step uu of row tile t) with their scale boxes, phase 1 two K steps of
// the down rows and their scale box; mp: the expert's six tensor maps.
template <int PH>
K3_DEV void mx_issue(uint32_t sbase, uint32_t full, int s, const CUtensorMap *mp, int uu, int t, uint64_t pol)
{
    using C = MxCfg<PH>;
    const uint32_t st = sbase + (uint32_t)(s * C::STAGE), sc = st + (uint32_t)(C::NMAT * C::A_BYTES);
    mbar_arrive_expect_tx(full, C::NMAT * C::A_BYTES + C::NSC * C::SC_BYTES);
    if (PH == 0) {
#pragma unroll
        for (int m = 0; m < 2; m++) {  // gate, up
            tma_load_2d_hint(st + (uint32_t)(m * C::A_BYTES), mp + m, uu * 128, t * MX_M, full, pol);
            tma_load_2d_hint(sc + (uint32_t)(m * C::SC_BYTES), mp + 3 + m, 16 * (uu >> 1), t * MX_M, full, pol);
        }
    } else {
#pragma unroll
        for (int m = 0; m < 2; m++)  // two K steps of the down rows
            tma_load_2d_hint(st + (uint32_t)(m * C::A_BYTES), mp + 2, (2 * uu + m) * 128, t * MX_M, full, pol);
        tma_load_2d_hint(sc, mp + 5, 16 * uu, t * MX_M, full, pol);
    }
}

// One wave of a phase on this CTA's share of its units.  sm: the
// 1024-aligned shared memory (phase layouts overlap: the phases run one after
// the other), bars: this phase's barriers, hready[j]: h tiles of expert slot j
// done.
template <int PH>
K3_DEV void mx_body(const MxArgs &a, uint8_t *sm, uint64_t *bars, uint32_t tmem, volatile int *abort_flag,
                    unsigned *s_last, unsigned *s_stop, unsigned *hready, const int32_t *sel_ids,
                    const float *sel_w, uint32_t prev_fin, const volatile unsigned *x_issued, const MxWave &w,
                    MxState<PH> &st, const uint64_t *prev_bars = nullptr, const uint32_t *prev_issued = nullptr)
{
    using C = MxCfg<PH>;
    using Bs = MxBars<PH>;
    constexpr int NMAT = C::NMAT, NS = C::NS;
    const uint32_t sbase = smem_addr(sm);
    const int K = PH == 0 ? a.d : a.f, ROWS = PH == 0 ? a.f : a.d;
    const uint32_t b_off = (uint32_t)(NS * C::STAGE);
    const uint32_t bimg_bytes = (uint32_t)K * 8u, bsf_bytes = (uint32_t)(K / 128) * 512u;
    const uint32_t sf_off = b_off + (PH == 0 ? bimg_bytes : 2 * bimg_bytes);
    const int B_FULL = Bs::FULL, B_AFULL = Bs::AFULL, B_EMPTY = Bs::EMPTY, B_ACCF = Bs::ACCF, B_ACCE = Bs::ACCE,
              B_BLOAD = Bs::BLOAD, B_BSCL = Bs::BSCL, B_FIN = Bs::FIN, B_BFREE = Bs::BFREE;
    auto bar = [&](int i) { return smem_addr(bars + i); };
    auto a_at = [&](int s, int m) { return sbase + (uint32_t)(s * C::STAGE + m * C::A_BYTES); };
    auto sc_at = [&](int s, int m) { return sbase + (uint32_t)(s * C::STAGE + NMAT * C::A_BYTES + m * C::SC_BYTES); };
    auto at_at = [&](int s, int m) {
        return sbase + (uint32_t)(s * C::STAGE + NMAT * C::A_BYTES + C::NSC * C::SC_BYTES + m * C::AT_BYTES);
    };
    constexpr int NOUT = C::NOUT;
    constexpr int EPI = PH == 0 ? MX_W_EPI : MX_W_EPI1;  // first of the phase's epilogue warps

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tpe = ROWS / MX_M;  // tiles per expert
    const int upt = K / C::UK;    // units per tile
    const int U = w.Uw, G = (int)gridDim.x;
    const int ulo = w.uw0 + U * (int)blockIdx.x / G, uhi = w.uw0 + U * ((int)blockIdx.x + 1) / G;
    // the CTA whose range holds unit u, and the end of CTA c's range
    auto cta_of = [&](int u) { return ((u - w.uw0 + 1) * G - 1) / U; };
    auto end_of = [&](int c) { return w.uw0 + U * (c + 1) / G; };

    // the experts of this CTA's range (phase 1 loads one B image per expert;
    // a range spans at most two experts, checked at launch)
    const int j_first = ulo < uhi ? (int)((ulo / upt) / tpe) : 0;
    const int j_last = ulo < uhi ? (int)(((uhi - 1) / upt) / tpe) : -1;

    if (warp == MX_W_PROD) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0 && ulo < uhi) {
            bool ok = true;
            // B operand images
            // phase 0: the x image copies were issued at the router's grid barrier
            uint32_t it = st.it;
            const uint64_t pol = l2_evict_first();  // weights: read once
            int cur_tile = -1;
            const CUtensorMap *mp = nullptr;
            int t = 0;
            for (int u = ulo + st.pre; u < uhi && ok && !*abort_flag; u++, it++) {
                const int tile = (int)(u / upt), uu = (int)(u % upt);
                if (tile != cur_tile) {
                    cur_tile = tile;
                    const int e = sel_ids[tile / tpe];
                    mp = a.maps + 6 * (size_t)e;
                    t = tile % tpe;
                }
                const int s = it % NS;
                if (it >= (uint32_t)NS && !tc_wait(bar(B_EMPTY + s), ((it / NS) - 1) & 1, a.err, abort_flag)) break;
                // phase 1 reuses phase 0's shared memory: the first fill of a
                // phase-1 stage waits until the MMAs of the phase-0 stages it
                // overlaps have read them for the last time (their final
                // `empty` phase), so the copies run on across the change of
                // phase; a stage reaching into phase 0's B image waits for all
                // of phase 0's MMAs
                if (PH == 1 && it < (uint32_t)NS && !mx_phase1_slot_free(s, prev_bars, prev_issued, prev_fin, a.err,
                                                                         abort_flag)) {
                    ok = false;
                    break;
                }
                // phase 0: the last stage holds the B scale atoms until they are in TMEM
                if (PH == 0 && it == (uint32_t)(NS - 1) && !tc_wait(bar(B_BSCL), 0, a.err, abort_flag)) {
                    ok = false;
                    break;
                }
                mx_issue<PH>(sbase, bar(B_FULL + s), s, mp, uu, t, pol);
                st.issued[s]++;
            }
            st.it = it;
            st.pre = 0;
        }
        if (lane == 0 && w.last) {
            // drain: every copy issued in this phase has landed before the CTA exits
            for (int s = 0; s < NS; s++)
                if (st.issued[s]) mbar_wait(bar(B_FULL + s), (st.issued[s] - 1) & 1, a.err);
            if (PH == 0 && *x_issued == 1u) mbar_wait(bar(B_BLOAD), 0, a.err);  // x image copies
        }
        __syncwarp();
    } else if (PH == 1 && warp == MX_W_BLD) {
        // ------------------------------- h pieces of this CTA's experts (phase 1)
        // once every h tile of expert slot j is written (acquire), bulk
        // copies into the next B buffer (the two buffers take a CTA's experts
        // in turn, across waves; a buffer is refilled once the MMAs of its
        // previous expert are done); the writers fenced their plain stores
        // towards the async proxy before publishing, the copy side does too
        if (lane == 0) {
            bool ok = !w.first || tc_wait(prev_fin, 0, a.err, abort_flag);  // phase 0's smem
            for (int x = 0; ulo < uhi && x <= j_last - j_first && ok && !*abort_flag; x++) {
                const int j = j_first + x;
                const int b = st.nexp & 1, use = st.nexp >> 1;
                if (use > 0 && !tc_wait(bar(B_BFREE + b), (use - 1) & 1, a.err, abort_flag)) break;
                if (!mx_wait_count(hready + j, (unsigned)(a.f / MX_M), a.err)) {  // h tiles of one expert
                    *abort_flag = 1;
                    break;
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_arrive_expect_tx(bar(B_BLOAD + b), bimg_bytes + bsf_bytes);
                for (uint32_t o = 0; o < bimg_bytes; o += 16384)
                    bulk_g2s(sbase + b_off + b * bimg_bytes + o, a.bimg + (size_t)j * bimg_bytes + o,
                             min(16384u, bimg_bytes - o), bar(B_BLOAD + b));
                bulk_g2s(sbase + sf_off + b * bsf_bytes, a.bsf + (size_t)j * bsf_bytes, bsf_bytes, bar(B_BLOAD + b));
                st.nexp++;
            }
            // drain: the copies land before the CTA exits (buffer b's last
            // fill is its ((nexp - b + 1) / 2)-th)
            if (w.last)
                for (int b = 0; b < 2 && b < st.nexp; b++)
                    mbar_wait(bar(B_BLOAD + b), (((st.nexp - b + 1) >> 1) - 1) & 1, a.err);
        }
        __syncwarp();
    } else if (ulo < uhi && warp == MX_W_PERM) {
        // ------------------------------------- scale boxes -> tcgen05.cp atoms
        // atom byte 16 r0 + 4 r1 + kb = scale of row r0 + 32 r1, k-block kb
        uint32_t it = st.it;
        for (int u = ulo; u < uhi && !*abort_flag; u++, it++) {
            const int uu = (int)(u % upt), s = it % NS;
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_FULL + s), (it / NS) & 1, a.err, abort_flag))) break;
#pragma unroll
            for (int m = 0; m < NMAT; m++)
#pragma unroll
                for (int at = 0; at < 2; at++)
#pragma unroll
                    for (int r1 = 0; r1 < 4; r1++) {
                        // phase 0: A tile m's own box, the unit's half; phase 1: the
                        // one box, tile m's half
                        const uint32_t box = PH == 0 ? sc_at(s, m) : sc_at(s, 0);
                        const int byte = PH == 0 ? 8 * (uu & 1) + 4 * at : 8 * m + 4 * at;
                        uint32_t v = lds32(box + (uint32_t)((lane + 32 * r1) * 16 + byte));
                        v &= ~__vcmpeq4(v, 0xffffffffu);  // 255 (a dropped group) -> 2^-127
                        sts32(at_at(s, m) + (uint32_t)(at * 512 + 16 * lane + 4 * r1), v);
                    }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_AFULL + s));
        }
        st.it = it;
    } else if (warp == MX_W_MMA) {
        // ------------------------------------------------------ MMA issuer
        bool ok = true;
        if (PH == 0 && w.first) {
            ok = __all_sync(0xffffffffu, tc_wait(bar(B_BLOAD), 0, a.err, abort_flag));
            if (ok) {
                tc_fence_after();
                for (int at = 0; at < K / 128; at++)
                    mx_cp_atom(tmem + C::TSB + 4 * at, sbase + (uint32_t)((NS - 1) * C::STAGE + 512 * at));
                mma_commit(bar(B_BSCL));
            }
        }
        uint32_t it = st.it, sg = st.sg;
        int bx = (st.nexp - 1) & 1;  // phase 1: B buffer of the current expert
        for (int u = ulo; u < uhi && ok && !*abort_flag; u++, it++) {
            const int tile = (int)(u / upt), uu = (int)(u % upt);
            const bool first = (u == ulo) || uu == 0, last = (u + 1 == uhi) || uu == upt - 1;
            if (PH == 1 && tile / tpe != st.cur_j) {
                // the previous expert's buffer is free once the MMAs issued so far are done
                if (st.cur_j >= 0) mma_commit(bar(B_BFREE + bx));
                st.cur_j = tile / tpe;
                bx = st.nexp & 1;
                const int use = st.nexp >> 1;
                st.nexp++;
                if (!__all_sync(0xffffffffu, tc_wait(bar(B_BLOAD + bx), use & 1, a.err, abort_flag))) break;
                tc_fence_after();
                for (int at = 0; at < K / 128; at++)
                    mx_cp_atom(tmem + C::TSB + (uint32_t)(bx * (K / 32) + 4 * at),
                               sbase + sf_off + (uint32_t)(bx * bsf_bytes + 512 * at));
            }
            const int buf = sg & 1;
            if (first && sg >= 2 &&
                !__all_sync(0xffffffffu, tc_wait(bar(B_ACCE + buf), ((sg / 2) - 1) & 1, a.err, abort_flag)))
                break;
            const int s = it % NS;
            if (!__all_sync(0xffffffffu, tc_wait(bar(B_AFULL + s), (it / NS) & 1, a.err, abort_flag))) break;
            tc_fence_after();
            const uint32_t tsa = tmem + C::TSA + (uint32_t)(s * NMAT * 8);
#pragma unroll
            for (int m = 0; m < NMAT; m++) {
                mx_cp_atom(tsa + m * 8, at_at(s, m));
                mx_cp_atom(tsa + m * 8 + 4, at_at(s, m) + 512);
            }
            const uint32_t bimg = sbase + b_off + (uint32_t)((PH == 1 ? bx : 0) * bimg_bytes);
            const uint32_t tsb = tmem + C::TSB + (uint32_t)((PH == 1 ? bx : 0) * (K / 32));
            if (PH == 0) {
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {
                    const int q = uu * 4 + q4;  // K step of 64 within the tile's K
                    const uint32_t blo = sw128_lo(bimg + (uint32_t)((q >> 2) * (MX_N * 128))) + 2u * (uint32_t)(q & 3);
                    const uint32_t idesc = mx_idesc(2u * (q4 & 1), 2u * (q & 1));
                    const uint32_t sfb = tsb + 4u * (uint32_t)(q >> 1);
#pragma unroll
                    for (int m = 0; m < 2; m++)  // gate, up: their own accumulators
                        mx_mma(tmem + (uint32_t)(C::TACC + buf * NOUT * MX_N + m * MX_N), sw128_lo(a_at(s, m)) + 2u * q4,
                               blo, idesc, tsa + m * 8 + 4 * (q4 >> 1), sfb, (first && q4 == 0) ? 0u : 1u);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 2; m++)  // the unit's two 256-long K steps, one accumulator
#pragma unroll
                    for (int q4 = 0; q4 < 4; q4++) {
                        const int q = uu * 8 + m * 4 + q4;
                        const uint32_t blo =
                            sw128_lo(bimg + (uint32_t)((q >> 2) * (MX_N * 128))) + 2u * (uint32_t)(q & 3);
                        const uint32_t idesc = mx_idesc(2u * (q4 & 1), 2u * (q & 1));
                        const uint32_t sfb = tsb + 4u * (uint32_t)(q >> 1);
                        mx_mma(tmem + (uint32_t)(C::TACC + buf * MX_N), sw128_lo(a_at(s, m)) + 2u * q4, blo, idesc,
                               tsa + m * 8 + 4 * (q4 >> 1), sfb, (first && m == 0 && q4 == 0) ? 0u : 1u);
                    }
            }
            mma_commit(bar(B_EMPTY + s));
            if (last) {
                mma_commit(bar(B_ACCF + buf));
                sg++;
            }
        }
        st.it = it;
        st.sg = sg;
        // every MMA and copy issued in this phase has completed before TMEM is freed
        if (w.last) {
            mma_commit(bar(B_FIN));
            mbar_wait(bar(B_FIN), 0, a.err);
        }
        __syncwarp();
    } else if (ulo < uhi && warp >= EPI && warp < EPI + 4) {
        // --------------------------------------------------------- epilogue
        // The four warps run the same segments and meet at the same named
        // barriers (bar 2): whether to go on is decided by one thread and
        // read by all between two barriers, so no warp can leave while the
        // others wait.
        const int qd = warp & 3, row = qd * 32 + lane;
        const bool leader = threadIdx.x == EPI * 32;
        uint32_t sg = st.sg;
        int u = ulo;
        int done_j[2] = {-1, -1}, done_n[2] = {0, 0};  // leader: h tiles finished per expert slot
        for (;;) {
            if (leader) *s_stop = (u >= uhi || *abort_flag) ? 1u : 0u;
            mx_bar_epi<PH>();
            const bool stop = *s_stop != 0u;
            mx_bar_epi<PH>();
            if (stop) break;
            const int tile = (int)(u / upt);
            const int t0 = tile * upt, t1 = t0 + upt;
            const int ua = u, ub = t1 < uhi ? t1 : uhi;
            u = ub;
            // a split tile's partial sums sit in slots indexed by the first
            // unit of their segment
            const bool whole = ua == t0 && ub == t1;
            const int seg = (int)(ua - t0);
            const int j = tile / tpe, t = tile % tpe;
            float pv[NOUT];
#pragma unroll
            for (int m = 0; m < NOUT; m++) pv[m] = 0.f;
            if (PH == 0 && !whole && ua == t0) {
                // the first segment: this CTA finishes the tile.  The other
                // segments' parts (published at the start of the other CTAs'
                // ranges) are waited for and read before this segment's own
                // accumulator is, so that their round trips overlap its MMAs;
                // they are added in unit order
                const float *pp = a.part + ((size_t)tile * upt) * MX_M * NOUT;
                int nother = 0;
                for (int us = ub; us < t1;) {
                    const int ub2 = end_of(cta_of(us));
                    us = ub2 < t1 ? ub2 : t1;
                    nother++;
                }
                if (leader) *s_last = mx_wait_count(a.cnt + tile, (unsigned)nother, a.err) ? 1u : 0u;
                __syncwarp();
                mx_bar_epi<PH>();
                if (*s_last != 1u) *abort_flag = 1;
                for (int us = ub; us < t1;) {
                    const int ub2 = end_of(cta_of(us)), ue = ub2 < t1 ? ub2 : t1;
#pragma unroll
                    for (int m = 0; m < NOUT; m++) pv[m] += __ldcg(pp + ((size_t)(us - t0) * MX_M + row) * NOUT + m);
                    us = ue;
                }
                if (leader) a.cnt[tile] = 0;  // for the next launch
            }
            const int buf = sg & 1;
            const bool ok = __all_sync(0xffffffffu, tc_wait(bar(B_ACCF + buf), (sg / 2) & 1, a.err, abort_flag));
            float v[NOUT];
#pragma unroll
            for (int m = 0; m < NOUT; m++) v[m] = 0.f;
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int m = 0; m < NOUT; m++) {
                    float c0[8], c1[8];
                    const uint32_t ta =
                        tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(C::TACC + buf * NOUT * MX_N + m * MX_N);
                    tmem_ld8(ta, c0);
                    tmem_ld8(ta + 8, c1);
                    tmem_wait_ld();
                    float acc = c1[7];  // the smallest pieces first
#pragma unroll
                    for (int i = 6; i >= 0; i--) acc += c1[i];
#pragma unroll
                    for (int i = 7; i >= 0; i--) acc += c0[i];
                    v[m] = acc;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_ACCE + buf));
            }
            sg++;
            if (PH == 0) {
                float *pp = a.part + ((size_t)tile * upt) * MX_M * NOUT;
                if (!whole && ua != t0) {
                    // a later segment: the CTA holding the tile's first units
                    // (at the end of its range, so it gets there last) finishes
                    // the tile; publish this part for it
#pragma unroll
                    for (int m = 0; m < NOUT; m++) pp[((size_t)seg * MX_M + row) * NOUT + m] = v[m];
                    __syncwarp();
                    mx_bar_epi<PH>();
                    if (leader) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.cnt + tile) : "memory");
                    continue;
                }
#pragma unroll
                for (int m = 0; m < NOUT; m++) v[m] += pv[m];
                const float h = silu(v[0]) * v[1];
                mx_encode_block(h, lane, (t * MX_M + qd * 32) / 32, a.himg + (size_t)j * a.f * 8,
                                a.hsf + (size_t)j * (a.f / 128) * 512);
                // h tiles done per expert slot, published together at the end
                if (leader) {
                    int q = 0;
                    while (q < 2 && done_j[q] >= 0 && done_j[q] != j) q++;
                    if (done_j[q] >= 0 && done_j[q] != j) {
                        set_device_error(a.err, K3MOE_EINVAL);  // a range spans at most two experts
                        *abort_flag = 1;
                    } else {
                        done_j[q] = j;
                        done_n[q]++;
                    }
                }
            } else {
                // w_j * (this segment's part of y_j) straight into out: the
                // down product is linear, so split tiles need no exchange
                red_add_f32(a.out + (size_t)t * MX_M + row, sel_w[j] * v[0]);
            }
        }
        st.sg = sg;
        if (PH == 0) {
            // every h piece this CTA wrote is in memory (and ordered towards
            // the async proxy that copies it) before the counts
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            mx_bar_epi<PH>();
            if (leader)
                for (int q = 0; q < 2; q++)
                    if (done_n[q])
                        asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(hready + done_j[q]),
                                     "r"((unsigned)done_n[q])
                                     : "memory");
        }
    }
}

// The producer's first NS - 1 units of phase 0's first wave, issued by the
// producer thread as soon as the experts are known (right after the top-k,
// before the code of the phase body is reached); the body's producer goes on
// from there.  Stage NS - 1 is left to it: that stage holds the B scale atoms
// until they are in TMEM.
K3_DEV void mx_preissue(const MxArgs &a, uint8_t *sm, uint64_t *bars, const int32_t *sel_ids, const MxWave &w,
                        MxState<0> &st)
{
    using C = MxCfg<0>;
    const int tpe = a.f / MX_M, upt = a.d / C::UK;
    const int U = w.Uw, G = (int)gridDim.x;
    const int ulo = w.uw0 + U * (int)blockIdx.x / G, uhi = w.uw0 + U * ((int)blockIdx.x + 1) / G;
    const uint64_t pol = l2_evict_first();
    int n = 0;
    for (int u = ulo; u < uhi && n < C::NS - 1; u++, n++) {
        const int tile = u / upt;
        mx_issue<0>(smem_addr(sm), smem_addr(bars + MxBars<0>::FULL + n), n, a.maps + 6 * (size_t)sel_ids[tile / tpe],
                    u % upt, tile % tpe, pol);
        st.issued[n]++;
    }
    st.it = (uint32_t)n;
    st.pre = n;
}

// Expert slots in a phase's first wave: three quarters of k (all of them for
// k < 4).  The second wave's gate/up time must cover the first wave's h
// epilogue, and the first wave's down time the second wave's.
K3_DEV int wave_split(int k) { return k < 4 ? k : (3 * k + 3) / 4; }

// Router of one token (phase R), spread over every CTA.
struct MxRoute {
    const void *x;          // [d] fp32 or bf16
    const uint16_t *Wr;     // [E][d] bf16
    Router rt;              // selection bias ([E] or null) and score rule
    float *logits;          // [E]
    uint8_t *ximg;          // pieces of x: B image, then scale atoms
    int32_t *ids_out;       // [k] selection (ascending ids), written by CTA 0
    float *w_out;           // [k] combine weights
    unsigned *gbar;         // grid barrier counter (zero between launches)
    int E;
};

// Phase R.  Each CTA copies its block of router rows (E / G rows, one
// contiguous piece of W_r) into its still unused stage memory with bulk
// copies (read once: evict-first in L2), and all its warps compute their
// logits from there, each over a slice of K; meanwhile warp g of the grid
// encodes 32-block g of x and the CTAs zero out.  A grid barrier, then every
// CTA reads the E logits and selects the top k itself while its last warp
// copies in the pieces of x.  False on a timeout.
template <typename XT>
K3_DEV bool mx_route(const MxRoute &r, const MxArgs &a0, float *out, uint8_t *sm, uint32_t bar_r, uint32_t bload0,
                     int32_t *sel_ids, float *s_logit, CtaTopkRedSmem &tk, unsigned *s_flag)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int d = a0.d, E = r.E, G = gridDim.x;
    const int e0 = (int)((long)E * blockIdx.x / G), e1 = (int)((long)E * (blockIdx.x + 1) / G);
    const uint32_t rowb = (uint32_t)d * 2u;  // one router row (<= 16 KB: d <= 8192)
    const uint32_t sbase = smem_addr(sm);
    if (threadIdx.x == 0) {
        // one copy and one barrier per row, so that a row's products start
        // as soon as it has landed
        const uint8_t *src = reinterpret_cast<const uint8_t *>(r.Wr + (size_t)e0 * d);
        const uint64_t pol = l2_evict_first();  // router rows: read once
        for (int q = 0; q < e1 - e0; q++) {
            mbar_arrive_expect_tx(bar_r + 8u * q, rowb);
            bulk_g2s_hint(sbase + rowb * q, src + (size_t)rowb * q, rowb, bar_r + 8u * q, pol);
        }
    }
    // Launched as a programmatic dependent of the previous kernel on the
    // stream: only the router rows (weights, never written by a kernel) are
    // requested before it has completed; x, out and the workspace are touched
    // after this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const XT *x = reinterpret_cast<const XT *>(r.x);
    const long NW = (long)G * (MX_THREADS / 32), gw = (long)blockIdx.x * (MX_THREADS / 32) + warp;
    const bool encodes = gw < (d >> 5);  // this warp writes pieces of x
    for (long b = gw; b < (d >> 5); b += NW) {
        float xv;
        if constexpr (sizeof(XT) == 4) xv = __ldg(reinterpret_cast<const float *>(x) + 32 * b + lane);
        else xv = __uint_as_float((uint32_t)__ldg(reinterpret_cast<const uint16_t *>(x) + 32 * b + lane) << 16);
        mx_encode_block(xv, lane, (int)b, r.ximg, r.ximg + (size_t)d * 8);
    }
    for (long i = (long)blockIdx.x * MX_THREADS + threadIdx.x; i < d; i += (long)G * MX_THREADS) out[i] = 0.f;
    // Logits of the CTA's rows, K-sliced: warp w takes 8-element chunks
    // [c0, c1) of every row (at most three per lane), so each lane reads its
    // x chunks once and keeps them in registers, and all warps work however
    // few rows the CTA holds; the warps' partial sums meet in shared memory
    // (s_logit, not yet in use) and are added in warp order.
    constexpr int NWR = MX_THREADS / 32;
    const int nr = e1 - e0;  // <= MX_ROUTER_ROWS, checked at launch
    const int nch = d >> 3, c0 = nch * warp / NWR, c1 = nch * (warp + 1) / NWR;
    float xr[3][8];
#pragma unroll
    for (int i = 0; i < 3; i++) {
        const int c = c0 + lane + 32 * i;
        if (c < c1) {
            load_x8<XT>(x, 8 * c, xr[i]);
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) xr[i][j] = 0.f;
        }
    }
    // (a loop, not unrolled over the row limit: the router runs once per
    // launch from cold instruction caches, where code size is time)
    bool ok = true;
#pragma unroll 1
    for (int q = 0; q < nr; q++) {
        float acc = 0.f;
        if (ok) ok = mbar_wait(bar_r + 8u * q, 0, a0.err);
        if (ok) {
            const uint32_t row = sbase + (uint32_t)q * rowb;
#pragma unroll
            for (int i = 0; i < 3; i++) {
                const int c = c0 + lane + 32 * i;
                if (c < c1) acc = bf16x8_dot(lds128(row + 16u * (uint32_t)c), xr[i], acc);
            }
        }
        const float v = warp_sum(acc);
        if (lane == 0) s_logit[warp * MX_ROUTER_ROWS + q] = v;
    }
    cta_sync_threads();
    if ((int)threadIdx.x < nr) {
        float l = 0.f;
        for (int w = 0; w < NWR; w++) l += s_logit[w * MX_ROUTER_ROWS + threadIdx.x];
        r.logits[e0 + threadIdx.x] = l;
    }
    // the x image is read by other CTAs' bulk copies (async proxy): its
    // writers order their stores towards that proxy
    if (encodes) asm volatile("fence.proxy.async.global;" ::: "memory");
    cta_sync_threads();
    if (threadIdx.x == 0) {
        bool good = ok;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(r.gbar) : "memory");
        good = mx_wait_count(r.gbar, G, a0.err) && good;
        *s_flag = good ? 1u : 0u;
    }
    cta_sync_threads();
    if (*s_flag != 1u) return false;
    if (threadIdx.x == (NWR - 1) * 32) {
        // phase 0's B operand, the pieces of x, while the top-k runs (in the
        // first eight warps): the image to its buffer, the scale atoms staged
        // in the last stage
        using C0 = MxCfg<0>;
        const uint32_t bimg = (uint32_t)d * 8u, bsf = (uint32_t)(d / 128) * 512u;
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(bload0, bimg + bsf);
        for (uint32_t o = 0; o < bimg; o += 16384)
            bulk_g2s(sbase + (uint32_t)(C0::NS * C0::STAGE) + o, r.ximg + o, min(16384u, bimg - o), bload0);
        for (uint32_t o = 0; o < bsf; o += 16384)
            bulk_g2s(sbase + (uint32_t)((C0::NS - 1) * C0::STAGE) + o, r.ximg + bimg + o, min(16384u, bsf - o),
                     bload0);
    }
    for (int e0b = threadIdx.x; e0b < E; e0b += 4 * MX_THREADS) {
        float v[4];
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int e = e0b + m * MX_THREADS;
            v[m] = e < E ? __ldcg(r.logits + e) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 4; m++) {
            const int e = e0b + m * MX_THREADS;
            if (e < E) s_logit[e] = v[m];
        }
    }
    cta_sync_threads();
    // the rule is a kernel parameter, the same in every thread: the default
    // softmax rule is passed as a constant so that its selection compiles
    // with the rule folded away
    auto logit_of = [&](int e) { return s_logit[e]; };
    if (r.rt.mode == K3_ROUTER_SOFTMAX)
        cta_topk_red(logit_of, Router{r.rt.bias, K3_ROUTER_SOFTMAX}, E, a0.k, sel_ids, tk,
                     [] { cta_sync_threads(); });
    else
        cta_topk_red(logit_of, r.rt, E, a0.k, sel_ids, tk, [] { cta_sync_threads(); });
    cta_sync_threads();
    if (blockIdx.x == 0 && threadIdx.x < a0.k) r.ids_out[threadIdx.x] = sel_ids[threadIdx.x];
    return true;
}

// The combine weights of the selected experts from their unbiased logits,
// by one warp (lane j < k: expert slot j), into sel_w and, from CTA 0, w_out.
K3_DEV void mx_weights(const MxRoute &r, int k, const int32_t *sel_ids, const float *s_logit, float *sel_w, int lane)
{
    const bool on = lane < k;
    const float w = router_weight(r.rt.mode, on ? s_logit[sel_ids[lane]] : 0.f, on);
    if (on) {
        sel_w[lane] = w;
        if (blockIdx.x == 0) r.w_out[lane] = w;
    }
}

// The whole layer for one token in one persistent kernel (one CTA per SM,
// all resident: CTAs wait for each other at the router's grid barrier and for
// the h tiles that other CTAs finish in phase 0).
template <typename XT>
__global__ void __launch_bounds__(MX_THREADS, 1)
    k3_mx_layer(const MxRoute r, const MxArgs a0, const MxArgs a1, unsigned *hready, unsigned *exit_cnt,
                uint32_t bar_off)
{
    __shared__ int32_t sel_ids[32];
    __shared__ float sel_w[32];
    __shared__ float s_logit[1024];
    __shared__ CtaTopkRedSmem tk;
    __shared__ unsigned s_flag;  // 1: the router's grid barrier passed, x image copies issued
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars0 = (uint64_t *)(sm + bar_off);
    uint64_t *bars1 = bars0 + MxBars<0>::N;
    uint64_t *bar_r = bars1 + MxBars<1>::N;  // router rows landed, one per row
    uint32_t *tmem_slot = (uint32_t *)(bar_r + MX_ROUTER_ROWS);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    unsigned *s_last = (unsigned *)(tmem_slot + 2);  // epilogue: this CTA completes the tile
    unsigned *s_stop = (unsigned *)(tmem_slot + 3);  // epilogue: no further segment
    unsigned *s_stop1 = (unsigned *)(tmem_slot + 4);  // the same for phase 1's epilogue warps
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        s_flag = 0;
        mx_init_bars<0>(bars0);
        mx_init_bars<1>(bars1);
        for (int q = 0; q < MX_ROUTER_ROWS; q++) mbar_init(smem_addr(bar_r + q), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MX_W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(MX_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)tmem_slot;

    if (!mx_route<XT>(r, a0, a1.out, sm, smem_addr(bar_r), smem_addr(bars0 + MxBars<0>::BLOAD), sel_ids, s_logit,
                      tk, &s_flag))
        *abort_flag = 1;
    cta_sync_threads();
    // Two waves per phase: gate/up of the first kA expert slots, then of the
    // rest; down of the first kA, then of the rest.  The first wave's h is
    // complete while the second wave's gate/up rows still stream, so the down
    // phase starts on h that is ready, and the second wave's h has the first
    // wave's down products to be finished in.
    const int kA = wave_split(a0.k), kB = a0.k - kA, nwave = kB > 0 ? 2 : 1;
    const int upe0 = (a0.f / MX_M) * (a0.d / MxCfg<0>::UK), upe1 = (a0.d / MX_M) * (a0.f / MxCfg<1>::UK);
    auto wave = [&](int wv, int upe) {
        return wv == 0 ? MxWave{0, kA * upe, true, nwave == 1} : MxWave{kA * upe, kB * upe, false, true};
    };
    MxState<0> st0;
    MxState<1> st1;
    if (warp == MX_W_PROD && (threadIdx.x & 31) == 0 && *abort_flag == 0)
        mx_preissue(a0, sm, bars0, sel_ids, wave(0, upe0), st0);
    // Each role goes on to phase 1 when it is done with phase 0; the roles
    // that write phase 1's shared memory (producer, h loader) first wait for
    // phase 0's MMAs to complete (its FIN barrier); phase 1's TMEM columns
    // are not phase 0's accumulators, which the epilogue may still read.
    const uint32_t fin0 = smem_addr(bars0 + MxBars<0>::FIN);
    // the next kernel on the stream may start its launch (its CTAs take
    // the SMs this grid leaves and wait for its completion before reading
    // anything it writes)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the combine weights are needed only by the phase-1 epilogue warps, whose
    // first named barrier orders them for the others of the four
    if (warp == MX_W_EPI1 && *abort_flag == 0) mx_weights(r, a0.k, sel_ids, s_logit, sel_w, threadIdx.x & 31);
    // The waves run in loops rather than as separate inlined bodies: the
    // kernel's code is far larger than the SM's instruction cache, and one
    // body per phase keeps it half as large (fewer instruction fetches from
    // L2 where the roles move on to new code).
#pragma unroll 1
    for (int wv = 0; wv < nwave; wv++)
        mx_body<0>(a0, sm, bars0, tmem, abort_flag, s_last, s_stop, hready, sel_ids, sel_w, 0u, &s_flag,
                   wave(wv, upe0), st0);
#pragma unroll 1
    for (int wv = 0; wv < nwave; wv++)
        mx_body<1>(a1, sm, bars1, tmem, abort_flag, s_last, s_stop1, hready, sel_ids, sel_w, fin0, &s_flag,
                   wave(wv, upe1), st1, bars0, st0.issued);

    tc_fence_before();
    cta_sync_threads();
    if (warp == MX_W_MMA) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(MX_TMEM_COLS)
                     : "memory");
    }
    // the last CTA out clears the h counters (no CTA reads them any more)
    if (threadIdx.x == 0 && ticket_add(exit_cnt, 1) == gridDim.x - 1) {
        for (int j = 0; j < a0.k; j++) hready[j] = 0;
        *r.gbar = 0;
        *exit_cnt = 0;
    }
}

// ---------------------------------------------------------------- host side

int num_sms();

bool mx_supported(int E, int k, int d, int f)
{
    // phase 0 stages the B scale atoms of x in one stage; TMEM holds d / 32
    // (phase 0) and 2 f / 32 (phase 1) columns of B scales
    return E >= 1 && k >= 1 && k <= 16 && d % 512 == 0 && f % 512 == 0 && d <= 8192 && f <= 2048 &&
           (d / 128) * 512 <= MxCfg<0>::STAGE && MxCfg<0>::TSB + d / 32 <= MX_TMEM_COLS &&
           MxCfg<1>::TSB + 2 * (f / 32) <= MX_TMEM_COLS && mx_smem(d, f) <= 232448;
}

// partial-sum slots: one per unit of a tile (a segment writes the slot of
// its first unit)
size_t mx_part_floats(int k, int d, int f) { return (size_t)k * (f / MX_M) * (d / MX_UK) * MX_M * 2; }
size_t mx_ximg_bytes(int d) { return (size_t)d * 8 + (size_t)(d / 128) * 512; }
size_t mx_himg_bytes(int k, int f) { return (size_t)k * ((size_t)f * 8 + (size_t)(f / 128) * 512); }
// counters: split phase-0 tiles' published parts, h tiles per expert slot, CTA exits, grid barrier
size_t mx_cnt_words(int k, int d, int f) { (void)d; return (size_t)k * (f / MX_M) + k + 2; }

// Tensor maps of E experts: [E][gate, up, down packed; gate, up, down scales]
// (packed: rows x in/2 bytes, boxes 128 rows x 128 bytes, 128-byte swizzle;
// scales: rows x in/32 bytes, boxes 128 rows x 16 bytes, no swizzle).
int mx_make_maps(const DevExpert *host_table, int E, int d, int f, void *dev_maps)
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
    CUtensorMap *maps = (CUtensorMap *)malloc(sizeof(CUtensorMap) * 6 * (size_t)E);
    if (!maps) return K3MOE_ENOMEM;
    int rc = K3MOE_OK;
    for (int e = 0; e < E && rc == K3MOE_OK; e++) {
        const uint8_t *planes[6] = {host_table[e].gp, host_table[e].up, host_table[e].dp,
                                    host_table[e].gs, host_table[e].us, host_table[e].ds};
        for (int m = 0; m < 6; m++) {
            const bool sc = m >= 3;
            const int rows = (m % 3) < 2 ? f : d, in = (m % 3) < 2 ? d : f;
            const cuuint64_t width = sc ? (cuuint64_t)(in / 32) : (cuuint64_t)(in / 2);
            const cuuint64_t dims[2] = {width, (cuuint64_t)rows};
            const cuuint64_t strides[1] = {width};
            const cuuint32_t box[2] = {sc ? 16u : 128u, (cuuint32_t)MX_M};
            const cuuint32_t estr[2] = {1, 1};
            if (encode(&maps[6 * e + m], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void *)planes[m], dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       sc ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
                rc = K3MOE_EINVAL;
                break;
            }
        }
    }
    if (rc == K3MOE_OK &&
        cudaMemcpy(dev_maps, maps, sizeof(CUtensorMap) * 6 * (size_t)E, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        rc = K3MOE_ECUDA;
    }
    free(maps);
    return rc;
}

// The whole batch-1 layer for one token: router and top-k (ids_out, w_out),
// gate/up + SwiGLU, down + weighted combine into out (overwritten).  x is
// fp32 or bf16 (xdt), logits / ximg / himg / part / cnt are the layer's
// workspace (cnt zero between launches).
template <typename XT>
static int launch_layer(const MxRoute &r, const MxArgs &a0, const MxArgs &a1, unsigned *hready, unsigned *exit_cnt,
                        uint32_t bar_off, size_t smem, cudaStream_t s)
{
    if (ensure_smem((const void *)k3_mx_layer<XT>, smem) != K3MOE_OK) return K3MOE_ECUDA;
    // The CTAs wait for each other (the router's grid barrier, the h tiles),
    // so all of them must be resident at once: one CTA per SM, and the SM
    // must hold one (checked once).  The launch is not a cooperative one: a
    // cooperative launch starts only when every SM is free at the same time,
    // which would keep it from the SMs that the previous kernel on the stream
    // leaves one by one.  Instead, where the driver takes it, it is a
    // programmatic dependent of that kernel, whose CTAs start as its CTAs exit
    // and request their router rows before it has completed.  Every wait
    // between CTAs is bounded, so a grid that could not become resident (an
    // SM held by other work for seconds) ends with K3MOE_ETIMEOUT in the
    // device error word rather than hanging.
    static std::atomic<int> resident{0};
    if (!resident.load(std::memory_order_relaxed)) {
        int b = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k3_mx_layer<XT>, MX_THREADS, smem) != cudaSuccess ||
            b < 1) {
            cudaGetLastError();
            return K3MOE_ECUDA;
        }
        resident.store(1, std::memory_order_relaxed);
    }
    static std::atomic<int> pdl_refused{0};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms());
    cfg.blockDim = dim3(MX_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_refused.load(std::memory_order_relaxed) ? 0 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k3_mx_layer<XT>, r, a0, a1, hready, exit_cnt, bar_off);
    if (e != cudaSuccess && cfg.numAttrs == 1) {
        cudaGetLastError();
        pdl_refused.store(1, std::memory_order_relaxed);
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, k3_mx_layer<XT>, r, a0, a1, hready, exit_cnt, bar_off);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ECUDA;
    }
    return K3MOE_OK;
}

int launch_mx_t1(const void *x, int xdt, const uint16_t *Wr, int E, Router rt, const void *maps,
                 float *logits, uint8_t *ximg, uint8_t *himg, float *part, unsigned *cnt, int k, int d, int f,
                 int32_t *ids_out, float *w_out, float *out, int *err, cudaStream_t s)
{
    const int G = num_sms();
    // phase 1 holds the B images of two experts: a CTA's range must not
    // span more than two; the in-kernel top-k takes E <= 1024
    const long upe1 = (long)(d / MX_M) * (f / MxCfg<1>::UK), u1 = (long)k * upe1;
    if ((u1 + G - 1) / G > upe1 || E > 1024) return K3MOE_EINVAL;
    // router rows below the stage holding the x scale atoms
    if ((size_t)((E + G - 1) / G) * d * 2 > (size_t)(MxCfg<0>::NS - 1) * MxCfg<0>::STAGE) return K3MOE_EINVAL;
    if ((E + G - 1) / G > MX_ROUTER_ROWS) return K3MOE_EINVAL;
    MxRoute r = {};
    r.x = x;
    r.Wr = Wr;
    r.rt = rt;
    r.logits = logits;
    r.ximg = ximg;
    r.ids_out = ids_out;
    r.w_out = w_out;
    r.E = E;
    MxArgs a0 = {};
    a0.maps = (const CUtensorMap *)maps;
    a0.k = k;
    a0.d = d;
    a0.f = f;
    a0.err = err;
    MxArgs a1 = a0;
    a0.bimg = ximg;
    a0.bsf = ximg + (size_t)d * 8;
    a0.himg = himg;
    a0.hsf = himg + (size_t)k * f * 8;
    a0.part = part;
    a0.cnt = cnt;
    a1.bimg = himg;
    a1.bsf = himg + (size_t)k * f * 8;
    a1.out = out;
    unsigned *hready = cnt + (size_t)k * (f / MX_M);
    unsigned *exit_cnt = hready + k;
    r.gbar = exit_cnt + 1;
    const uint32_t bar_off = (uint32_t)mx_bar_off(d, f);
    const size_t smem = mx_smem(d, f);
    if (xdt == K3MOE_F32) return launch_layer<float>(r, a0, a1, hready, exit_cnt, bar_off, smem, s);
    if (xdt == K3MOE_BF16) return launch_layer<__nv_bfloat16>(r, a0, a1, hready, exit_cnt, bar_off, smem, s);
    return K3MOE_EINVAL;
}

}  // namespace k3
