// k3_capi.cu -- the extern "C" entry points of k3moe.h: argument checks,
// library-owned layer scratch, and the launch sequence of each call.
#include <cuda_runtime.h>

#include <algorithm>

#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "k3_device.cuh"

namespace k3 {
int num_sms();

int launch_rows_t1(int mode, const float *x, const ExpertSrc &src, int k, int in, int rows,
                   float *out, cudaStream_t s);
int launch_down_t1(const float *h, const ExpertSrc &src, const float *w, int k, int d, int f,
                   float *out, cudaStream_t s, bool acc = false);
int route_t1_splits(int d);
int launch_route_t1(const void *x, int xdt, const uint16_t *Wr, int E, int d, float *part,
                    float *logits, Router rt, int k, int32_t *ids, float *w,
                    unsigned *ticket, float eps, float *u, cudaStream_t s);
bool mx_supported(int E, int k, int d, int f);
size_t mx_part_floats(int k, int d, int f);
size_t mx_ximg_bytes(int d);
size_t mx_himg_bytes(int k, int f);
size_t mx_cnt_words(int k, int d, int f);
int mx_make_maps(const DevExpert *host_table, int E, int d, int f, void *dev_maps);
int launch_mx_t1(const void *x, int xdt, const uint16_t *Wr, int E, Router rt, const void *maps,
                 float *logits, uint8_t *ximg, uint8_t *himg, float *part, unsigned *cnt, int k, int d, int f,
                 int32_t *ids_out, float *w_out, float *out, int *err, cudaStream_t s);
int route_multi_nsplit(int T, int E, int d);
int launch_route_multi(const void *X, int xdt, int T, const uint16_t *Wr, int E, int d,
                       float *part, int nsplit, float *logits, Router rt, int k,
                       int32_t *ids, float *w, cudaStream_t s);
int launch_group(const int32_t *ids, int npairs, int E, int nt, int32_t *offsets, int32_t *perm,
                 int4 *items, int32_t *n_items, cudaStream_t s);
int grouped_nt();
bool tc_supported(int E, int k, int d, int f);
bool mxq_supported(int E, int k, int d, int f);
bool shared_supported(int n, int d, int f);
size_t shared_workspace_floats(int n, int f);
int launch_shared(const uint16_t *const *gate, const uint16_t *const *up, const uint16_t *const *down, int n,
                  const float *x, int T, int d, int f, float *h, float *out, int accumulate, cudaStream_t s);
int mxq_max_tiles(int npairs, int E);
size_t mxq_max_rows(int npairs, int E);
size_t mxq_tile_bytes();
int launch_mx_quantize(const void *x, int xdt, int rows, int cols, uint8_t *codes, uint8_t *scales,
                       cudaStream_t s);
int launch_mxq_gateup(const void *X, int xdt, int T, int k, int E, int d, int f, const void *maps,
                      const int32_t *offsets, const int32_t *perm, void *tiles, int32_t *n_tiles, int32_t *tbase,
                      int32_t *slot, int max_tiles, uint8_t *Xg, uint8_t *Xsf, uint8_t *Hg, uint8_t *Hsf, int *err,
                      cudaStream_t s);
int launch_mxq_down(int T, int k, int d, int f, const void *maps, const int32_t *perm, const float *wsel,
                    const void *tiles, const int32_t *n_tiles, const uint8_t *Hg, const uint8_t *Hsf, float *out,
                    int *err, cudaStream_t s);
int tc_max_tiles(int npairs, int E);
size_t tc_xg_bytes(int npairs, int E, int d);
size_t tc_hg_bytes(int npairs, int E, int f);
size_t tc_tile_bytes();
size_t tc_map_bytes();
int tc_make_maps(const DevExpert *host_table, int E, int d, int f, void *dev_maps);
int tc_e4m3_eligible(const DevExpert *dev_table, int E, int d, int f, cudaStream_t s);
int launch_tc_gateup(const void *X, int xdt, int T, int kd, int k, int E, int d, int f, const DevExpert *table,
                     const void *maps, const int32_t *offsets, const int32_t *perm, void *tiles, int32_t *n_tiles,
                     int max_tiles, float *tscale, uint8_t *Xg, uint8_t *Hg, float *hf, unsigned *hmax, int *err,
                     cudaStream_t s);
int launch_tc_down(int T, int kd, int k, int d, int f, const DevExpert *table, const void *maps, const int32_t *perm,
                   const float *wsel, const void *tiles, const int32_t *n_tiles, uint8_t *Hg, const float *hf,
                   unsigned *hmax, float *out, int *err, cudaStream_t s);
int launch_grouped_gateup(const void *X, int xdt, const DevExpert *table, const int32_t *perm,
                          const int4 *items, const int32_t *n_items, int max_items, int k, int d,
                          int f, float *h, cudaStream_t s);
int launch_grouped_down(const float *h, const DevExpert *table, const int32_t *perm,
                        const int4 *items, const int32_t *n_items, int max_items, int k, int d,
                        int f, const float *wsel, float *Y, cudaStream_t s);
int launch_combine(const float *Y, int T, int k, int d, float *out, cudaStream_t s);
int launch_rmsnorm(float *u, const float *x, int n, float eps, cudaStream_t s);
int launch_residual(float *x, const float *dlt, int n, cudaStream_t s);
bool fused_t1_supported(int E, int k, int d, int f);
int launch_fused_t1(const float *x, const uint16_t *Wr, Router rt, const DevExpert *table,
                    int E, int k, int d, int f, float *logits, int32_t *ids, float *w, float *h,
                    float *Y, float *out, unsigned long long *ctr, bool act16, cudaStream_t s);
int fused_t1_counters();
}  // namespace k3

using k3::DevExpert;
using k3::ExpertSrc;

#define K3_TRY(expr)                 \
    do {                             \
        int _st = (expr);            \
        if (_st != K3MOE_OK) return _st; \
    } while (0)
#define K3_CUDA(expr)                                     \
    do {                                                  \
        if ((expr) != cudaSuccess) {                      \
            cudaGetLastError();                           \
            return K3MOE_ECUDA;                           \
        }                                                 \
    } while (0)

static inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static inline cudaStream_t cs(k3moe_stream s) { return reinterpret_cast<cudaStream_t>(s); }

static bool valid_dims(int32_t d, int32_t f)
{
    return d > 0 && f > 0 && d % 32 == 0 && f % 32 == 0 && d <= 16384 && f <= 2048;
}

static bool valid_mat(const k3moe_mat &m, int rows, int in)
{
    return m.packed && m.scales && aligned16(m.packed) && aligned16(m.scales) && m.rows == rows &&
           m.in == in;
}

static bool valid_expert(const k3moe_expert &e, int d, int f)
{
    return valid_mat(e.gate, f, d) && valid_mat(e.up, f, d) && valid_mat(e.down, d, f);
}

static DevExpert to_dev(const k3moe_expert &e)
{
    DevExpert x;
    x.gp = e.gate.packed;
    x.gs = e.gate.scales;
    x.up = e.up.packed;
    x.us = e.up.scales;
    x.dp = e.down.packed;
    x.ds = e.down.scales;
    return x;
}

extern "C" {

const char *k3moe_strerror(int st)
{
    switch (st) {
    case K3MOE_OK: return "ok";
    case K3MOE_EINVAL: return "invalid argument";
    case K3MOE_ENOMEM: return "out of memory";
    case K3MOE_ECUDA: return "CUDA runtime error";
    case K3MOE_ETIMEOUT: return "bounded wait timed out";
    case K3MOE_EBUSY: return "no evictable cache slot";
    case K3MOE_ENODEV: return "no usable device";
    case K3MOE_EIO: return "file input/output error";
    default: return "unknown status";
    }
}

int k3moe_version(void) { return (1 << 16) | 0; }

int k3moe_device_error(void)
{
    int *word = k3::device_error_word();
    if (!word) return K3MOE_ECUDA;
    int v = 0;
    K3_CUDA(cudaDeviceSynchronize());
    K3_CUDA(cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost));
    K3_CUDA(cudaMemset(word, 0, sizeof(int)));
    return v;
}

int64_t k3moe_matrix_bytes(int32_t rows, int32_t in)
{
    if (rows <= 0 || in <= 0 || in % 32) return -1;
    return (int64_t)rows * (in / 2 + in / 32);
}

int64_t k3moe_expert_bytes(int32_t d, int32_t f)
{
    if (d <= 0 || f <= 0 || d % 32 || f % 32) return -1;
    return 2 * k3moe_matrix_bytes(f, d) + k3moe_matrix_bytes(d, f);
}

int k3moe_expert_view(k3moe_expert *out, const void *blob, int32_t d, int32_t f)
{
    if (!out || !blob || d <= 0 || f <= 0 || d % 32 || f % 32 || !aligned16(blob))
        return K3MOE_EINVAL;
    const uint8_t *b = (const uint8_t *)blob;
    const size_t gpB = (size_t)f * d / 2, gsB = (size_t)f * d / 32;
    const size_t dpB = (size_t)d * f / 2;
    out->gate = {b, b + gpB, f, d};
    b += gpB + gsB;
    out->up = {b, b + gpB, f, d};
    b += gpB + gsB;
    out->down = {b, b + dpB, d, f};
    return K3MOE_OK;
}

int k3moe_pack_expert(void *blob, const uint8_t *gp, const uint8_t *gs, const uint8_t *up,
                      const uint8_t *us, const uint8_t *dp, const uint8_t *ds, int32_t d,
                      int32_t f, k3moe_stream s)
{
    k3moe_expert v;
    K3_TRY(k3moe_expert_view(&v, blob, d, f));
    if (!gp || !gs || !up || !us || !dp || !ds) return K3MOE_EINVAL;
    const size_t pB = (size_t)f * d / 2, sB = (size_t)f * d / 32;
    K3_CUDA(cudaMemcpyAsync((void *)v.gate.packed, gp, pB, cudaMemcpyDefault, cs(s)));
    K3_CUDA(cudaMemcpyAsync((void *)v.gate.scales, gs, sB, cudaMemcpyDefault, cs(s)));
    K3_CUDA(cudaMemcpyAsync((void *)v.up.packed, up, pB, cudaMemcpyDefault, cs(s)));
    K3_CUDA(cudaMemcpyAsync((void *)v.up.scales, us, sB, cudaMemcpyDefault, cs(s)));
    K3_CUDA(cudaMemcpyAsync((void *)v.down.packed, dp, pB, cudaMemcpyDefault, cs(s)));
    K3_CUDA(cudaMemcpyAsync((void *)v.down.scales, ds, sB, cudaMemcpyDefault, cs(s)));
    return K3MOE_OK;
}

int k3moe_matmul_mxfp4(float *y, const float *x, const k3moe_mat *W, k3moe_stream s)
{
    if (!y || !x || !W || !W->packed || !W->scales) return K3MOE_EINVAL;
    if (W->rows <= 0 || W->in <= 0 || W->in % 32 || W->in > 16384) return K3MOE_EINVAL;
    if (!aligned16(y) || !aligned16(x) || !aligned16(W->packed) || !aligned16(W->scales))
        return K3MOE_EINVAL;
    ExpertSrc src;
    memset(&src, 0, sizeof(src));
    src.inl[0].gp = W->packed;
    src.inl[0].gs = W->scales;
    return k3::launch_rows_t1(0, x, src, 1, W->in, W->rows, y, cs(s));
}

size_t k3moe_expert_gemv_workspace(int32_t d, int32_t f)
{
    if (!valid_dims(d, f)) return 0;
    return (size_t)f * sizeof(float);
}

int k3moe_expert_gemv(float *y, const float *x, const k3moe_expert *e, int32_t d, int32_t f,
                      void *ws, size_t ws_bytes, k3moe_stream s)
{
    if (!y || !x || !e || !ws || !valid_dims(d, f) || !valid_expert(*e, d, f)) return K3MOE_EINVAL;
    if (!aligned16(y) || !aligned16(x) || !aligned16(ws) ||
        ws_bytes < k3moe_expert_gemv_workspace(d, f))
        return K3MOE_EINVAL;
    ExpertSrc src;
    memset(&src, 0, sizeof(src));
    src.inl[0] = to_dev(*e);
    float *h = (float *)ws;
    K3_TRY(k3::launch_rows_t1(1, x, src, 1, d, f, h, cs(s)));
    return k3::launch_down_t1(h, src, nullptr, 1, d, f, y, cs(s));
}

}  // extern "C"

// ------------------------------------------------------------------ layer

struct k3moe_layer {
    int E, k, d, f, maxT;
    const uint16_t *Wr;
    const float *bias;
    DevExpert *table;    // [E]
    float *logits;       // [maxT * E]
    float *part;         // [nsplit * maxT * E]
    int nsplit;
    int32_t *ids;        // [maxT * k]
    float *w;            // [maxT * k]
    float *h;            // [maxT * k * f]
    float *Y;            // [maxT * k * d]  (T > 1)
    int32_t *offsets;    // [E + 1]
    int32_t *perm;       // [maxT * k]
    int4 *items;         // [maxT * k]
    int32_t *n_items;    // [1]
    unsigned *ticket;    // [1]
    cudaEvent_t ev[4];   // optional timing events (caller-owned)
    int nev;
    bool router_only;    // created without a resident expert table
    bool fused;          // K3MOE_OPT_FUSED_T1
    bool act16;          // K3MOE_OPT_ACT_F16
    bool sigmoid;        // K3MOE_OPT_SIGMOID_ROUTER
    bool sig_norm;       // K3MOE_OPT_SIGMOID_NORM
    unsigned long long *ctr;  // monotonic cross-CTA counters of the fused kernel
    // tensor-core grouped path (T > 1)
    bool tc;             // K3MOE_OPT_TC (default on where supported)
    bool tc_ready;       // its buffers and tensor maps exist
    void *tc_tiles;      // [tc_max_tiles] tiles
    int32_t *tc_ntiles;  // [1]
    int tc_max_tiles;
    uint8_t *Xg;         // token rows, bf16, tile-major
    uint8_t *Hg;         // SwiGLU rows (hi, lo), bf16, tile-major
    void *tc_maps;       // [E][3] tensor maps of the packed planes
    bool e4m3_ok;        // every gate/up scale byte allows the exact e4m3 decode
    bool e4m3;           // K3MOE_OPT_TC_E4M3 (default on where e4m3_ok)
    float *tscale;       // [maxT] token scales of the e4m3 pieces
    float *hf;           // [maxT * k * f] h in fp32 (e4m3 down)
    unsigned *hmax;      // [maxT * k] per-pair max |h| bits (e4m3 down)
    // block-scaled tensor-core path of one token (kind::mxf4)
    bool mx;             // K3MOE_OPT_MX (default on where supported)
    bool mx_ready;       // its buffers and tensor maps exist
    void *mx_maps;       // [E][6] tensor maps: packed and scale planes
    uint8_t *mx_ximg;    // pieces of x: B image + scale atoms
    uint8_t *mx_himg;    // pieces of h per selected expert
    float *mx_part;      // split-tile partial sums
    // MXFP4-activation grouped path (T > 1, kind::mxf4)
    bool mxq;            // K3MOE_OPT_MXQ (default off)
    bool mxq_ready;      // its buffers exist (and the mx tensor maps)
    void *mq_tiles;      // [mq_max_tiles] tiles
    int32_t *mq_ntiles;  // [1]
    int32_t *mq_tbase;   // [E] first tile of each expert
    int32_t *mq_slot;    // [maxT * k] tile row of each pair
    int mq_max_tiles;
    uint8_t *mq_xg, *mq_xsf;  // token codes (rows) and scale atoms (per tile)
    uint8_t *mq_hg, *mq_hsf;  // h codes and scale atoms
    unsigned *mx_cnt;    // tile tickets (zero between launches)
};

// The layer's selection rule: its bias and score rule (K3MOE_OPT_SIGMOID_*).
static k3::Router router_of(const k3moe_layer *L)
{
    return k3::Router{L->bias, L->sigmoid ? (L->sig_norm ? k3::K3_ROUTER_SIGMOID_NORM : k3::K3_ROUTER_SIGMOID)
                                         : k3::K3_ROUTER_SOFTMAX};
}

static void layer_free(k3moe_layer *L)
{
    if (!L) return;
    void *ptrs[] = {L->table, L->logits, L->part,  L->ids,     L->w,      L->h,    L->Y,
                    L->offsets, L->perm, L->items, L->n_items, L->ticket, L->ctr,
                    L->tc_tiles, L->tc_ntiles, L->Xg, L->Hg, L->tc_maps, L->tscale, L->hf, L->hmax,
                    L->mx_maps, L->mx_ximg, L->mx_himg, L->mx_part, L->mx_cnt,
                    L->mq_tiles, L->mq_ntiles, L->mq_tbase, L->mq_slot, L->mq_xg, L->mq_xsf, L->mq_hg, L->mq_hsf};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    delete L;
}

extern "C" {

int k3moe_layer_create(k3moe_layer **out, const k3moe_layer_desc *D)
{
    if (!out || !D) return K3MOE_EINVAL;
    *out = nullptr;
    if (D->n_experts <= 0 || D->n_experts > 1024 || D->top_k <= 0 || D->top_k > 16 || D->top_k > D->n_experts ||
        !valid_dims(D->d, D->f) || !D->router_w || D->max_tokens <= 0 ||
        !aligned16(D->router_w) || (D->sel_bias && ((uintptr_t)D->sel_bias & 3u)))
        return K3MOE_EINVAL;
    if (D->host_experts)
        for (int e = 0; e < D->n_experts; e++)
            if (!valid_expert(D->host_experts[e], D->d, D->f)) return K3MOE_EINVAL;
    if (!k3::device_error_word()) return K3MOE_ECUDA;  // look the word up before any capture
    k3moe_layer *L = new (std::nothrow) k3moe_layer;
    if (!L) return K3MOE_ENOMEM;
    memset(L, 0, sizeof(*L));
    L->E = D->n_experts;
    L->k = D->top_k;
    L->d = D->d;
    L->f = D->f;
    L->maxT = D->max_tokens;
    L->Wr = D->router_w;
    L->bias = D->sel_bias;
    L->nsplit = k3::route_multi_nsplit(L->maxT, L->E, L->d);
    const size_t pairs = (size_t)L->maxT * L->k;
    bool ok = true;
    auto alloc = [&](void **p, size_t bytes) {
        if (ok && cudaMalloc(p, bytes ? bytes : 16) != cudaSuccess) {
            cudaGetLastError();
            ok = false;
        }
    };
    alloc((void **)&L->table, sizeof(DevExpert) * L->E);
    alloc((void **)&L->logits, sizeof(float) * L->maxT * L->E);
    // multi-token split-K partials, or the batch-1 router's [S][E] partials + S sums of x^2
    const size_t t1part = (size_t)k3::route_t1_splits(L->d) * (L->E + 1);
    alloc((void **)&L->part, sizeof(float) * std::max((size_t)L->nsplit * L->maxT * L->E, t1part));
    alloc((void **)&L->ids, sizeof(int32_t) * pairs);
    alloc((void **)&L->w, sizeof(float) * pairs);
    alloc((void **)&L->h, sizeof(float) * pairs * L->f);
    alloc((void **)&L->Y, sizeof(float) * pairs * L->d);
    alloc((void **)&L->offsets, sizeof(int32_t) * (L->E + 1));
    alloc((void **)&L->perm, sizeof(int32_t) * pairs);
    alloc((void **)&L->items, sizeof(int4) * pairs);
    alloc((void **)&L->n_items, sizeof(int32_t));
    alloc((void **)&L->ticket, sizeof(unsigned));
    alloc((void **)&L->ctr, sizeof(unsigned long long) * k3::fused_t1_counters());
    if (L->maxT > 1 && D->host_experts && k3::tc_supported(L->E, L->k, L->d, L->f)) {
        L->tc_max_tiles = k3::tc_max_tiles((int)pairs, L->E);
        alloc(&L->tc_tiles, k3::tc_tile_bytes() * L->tc_max_tiles);
        alloc((void **)&L->tc_ntiles, sizeof(int32_t));
        alloc((void **)&L->Xg, k3::tc_xg_bytes((int)pairs, L->E, L->d));
        alloc((void **)&L->Hg, k3::tc_hg_bytes((int)pairs, L->E, L->f));
        alloc((void **)&L->tscale, sizeof(float) * L->maxT);
        alloc((void **)&L->hf, sizeof(float) * pairs * L->f);
        alloc((void **)&L->hmax, sizeof(unsigned) * pairs);
        alloc(&L->tc_maps, k3::tc_map_bytes() * 3 * L->E);
        L->tc_ready = ok;
        L->tc = true;
    }
    if (D->host_experts && k3::mx_supported(L->E, L->k, L->d, L->f)) {
        alloc(&L->mx_maps, k3::tc_map_bytes() * 6 * L->E);
        alloc((void **)&L->mx_ximg, k3::mx_ximg_bytes(L->d));
        alloc((void **)&L->mx_himg, k3::mx_himg_bytes(L->k, L->f));
        alloc((void **)&L->mx_part, sizeof(float) * k3::mx_part_floats(L->k, L->d, L->f));
        alloc((void **)&L->mx_cnt, sizeof(unsigned) * k3::mx_cnt_words(L->k, L->d, L->f));
        L->mx_ready = ok;
        L->mx = true;
        if (L->maxT > 1 && k3::mxq_supported(L->E, L->k, L->d, L->f)) {
            L->mq_max_tiles = k3::mxq_max_tiles((int)pairs, L->E);
            const size_t rows = k3::mxq_max_rows((int)pairs, L->E);
            alloc(&L->mq_tiles, k3::mxq_tile_bytes() * L->mq_max_tiles);
            alloc((void **)&L->mq_ntiles, sizeof(int32_t));
            alloc((void **)&L->mq_tbase, sizeof(int32_t) * L->E);
            alloc((void **)&L->mq_slot, sizeof(int32_t) * pairs);
            alloc((void **)&L->mq_xg, rows * (L->d / 2));
            alloc((void **)&L->mq_xsf, (size_t)L->mq_max_tiles * (L->d / 128) * 512);
            alloc((void **)&L->mq_hg, rows * (L->f / 2));
            alloc((void **)&L->mq_hsf, (size_t)L->mq_max_tiles * (L->f / 128) * 512);
            L->mxq_ready = ok;
        }
    }
    L->fused = true;
    L->act16 = false;
    if (!ok) {
        layer_free(L);
        return K3MOE_ENOMEM;
    }
    DevExpert *tmp = (DevExpert *)malloc(sizeof(DevExpert) * L->E);
    if (!tmp) {
        layer_free(L);
        return K3MOE_ENOMEM;
    }
    for (int e = 0; e < L->E; e++) {
        if (D->host_experts)
            tmp[e] = to_dev(D->host_experts[e]);
        else
            memset(&tmp[e], 0, sizeof(DevExpert));
    }
    L->router_only = D->host_experts == nullptr;
    cudaError_t st = cudaMemcpy(L->table, tmp, sizeof(DevExpert) * L->E, cudaMemcpyHostToDevice);
    if (st == cudaSuccess && L->tc_ready && k3::tc_make_maps(tmp, L->E, L->d, L->f, L->tc_maps) != K3MOE_OK)
        L->tc_ready = false;  // the CUDA-core grouped path serves instead
    if (st == cudaSuccess && L->tc_ready) {
        L->e4m3_ok = k3::tc_e4m3_eligible(L->table, L->E, L->d, L->f, 0) == 1;
        L->e4m3 = L->e4m3_ok;
    }
    if (st == cudaSuccess && L->mx_ready) {
        if (k3::mx_make_maps(tmp, L->E, L->d, L->f, L->mx_maps) != K3MOE_OK) {
            L->mx_ready = false;  // the fused CUDA-core kernel serves instead
            L->mxq_ready = false;
        } else {
            st = cudaMemset(L->mx_cnt, 0, sizeof(unsigned) * k3::mx_cnt_words(L->k, L->d, L->f));
            if (st == cudaSuccess) st = cudaMemset(L->mx_ximg, 0, k3::mx_ximg_bytes(L->d));
            if (st == cudaSuccess) st = cudaMemset(L->mx_himg, 0, k3::mx_himg_bytes(L->k, L->f));
        }
    }
    free(tmp);
    if (st == cudaSuccess) st = cudaMemset(L->ticket, 0, sizeof(unsigned));
    if (st == cudaSuccess)
        st = cudaMemset(L->ctr, 0, sizeof(unsigned long long) * k3::fused_t1_counters());
    if (st != cudaSuccess) {
        cudaGetLastError();
        layer_free(L);
        return K3MOE_ECUDA;
    }
    *out = L;
    return K3MOE_OK;
}

int k3moe_layer_destroy(k3moe_layer *L)
{
    if (!L) return K3MOE_EINVAL;
    layer_free(L);
    return K3MOE_OK;
}

static int route_into(k3moe_layer *L, const void *X, int xdt, int32_t T, cudaStream_t s)
{
    if (T == 1)
        return k3::launch_route_t1(X, xdt, L->Wr, L->E, L->d, L->part, L->logits, router_of(L), L->k,
                                   L->ids, L->w, L->ticket, 0.f, nullptr, s);
    return k3::launch_route_multi(X, xdt, T, L->Wr, L->E, L->d, L->part, L->nsplit, L->logits,
                                  router_of(L), L->k, L->ids, L->w, s);
}

static bool valid_call(k3moe_layer *L, const void *X, int xdt, int32_t T)
{
    return L && X && aligned16(X) && (xdt == K3MOE_F32 || xdt == K3MOE_BF16) && T >= 1 &&
           T <= L->maxT;
}

int k3moe_layer_route(k3moe_layer *L, const void *X, int xdt, int32_t T, int32_t *ids, float *w,
                      k3moe_stream s)
{
    if (!valid_call(L, X, xdt, T) || !ids || !w) return K3MOE_EINVAL;
    K3_TRY(route_into(L, X, xdt, T, cs(s)));
    K3_CUDA(cudaMemcpyAsync(ids, L->ids, sizeof(int32_t) * T * L->k, cudaMemcpyDeviceToDevice,
                            cs(s)));
    K3_CUDA(cudaMemcpyAsync(w, L->w, sizeof(float) * T * L->k, cudaMemcpyDeviceToDevice, cs(s)));
    return K3MOE_OK;
}

int k3moe_layer_forward(k3moe_layer *L, const void *X, int xdt, int32_t T, float *out,
                        int32_t *ids_out, float *w_out, k3moe_stream s)
{
    if (!valid_call(L, X, xdt, T) || !out || !aligned16(out) || L->router_only)
        return K3MOE_EINVAL;
    cudaStream_t st = cs(s);
    if (L->nev) K3_CUDA(cudaEventRecord(L->ev[0], st));
    if (T == 1 && L->mx && L->mx_ready) {
        // one persistent kernel: router and top-k, then the block-scaled
        // gate/up and down phases
        K3_TRY(k3::launch_mx_t1(X, xdt, L->Wr, L->E, router_of(L), L->mx_maps, L->logits, L->mx_ximg, L->mx_himg,
                                L->mx_part, L->mx_cnt, L->k, L->d, L->f, L->ids, L->w, out,
                                k3::device_error_word(), st));
        if (L->nev) {
            K3_CUDA(cudaEventRecord(L->ev[1], st));
            K3_CUDA(cudaEventRecord(L->ev[2], st));
            K3_CUDA(cudaEventRecord(L->ev[3], st));
        }
        if (ids_out)
            K3_CUDA(cudaMemcpyAsync(ids_out, L->ids, sizeof(int32_t) * L->k, cudaMemcpyDeviceToDevice, st));
        if (w_out) K3_CUDA(cudaMemcpyAsync(w_out, L->w, sizeof(float) * L->k, cudaMemcpyDeviceToDevice, st));
        return K3MOE_OK;
    }
    if (T == 1 && xdt == K3MOE_F32 && k3moe_layer_fused_t1(L) == 1) {
        K3_TRY(k3::launch_fused_t1((const float *)X, L->Wr, router_of(L), L->table, L->E, L->k, L->d,
                                   L->f, L->logits, L->ids, L->w, L->h, L->Y, out, L->ctr,
                                   L->act16, st));
        if (L->nev) {
            K3_CUDA(cudaEventRecord(L->ev[1], st));
            K3_CUDA(cudaEventRecord(L->ev[2], st));
            K3_CUDA(cudaEventRecord(L->ev[3], st));
        }
        if (ids_out)
            K3_CUDA(cudaMemcpyAsync(ids_out, L->ids, sizeof(int32_t) * L->k,
                                    cudaMemcpyDeviceToDevice, st));
        if (w_out)
            K3_CUDA(cudaMemcpyAsync(w_out, L->w, sizeof(float) * L->k, cudaMemcpyDeviceToDevice,
                                    st));
        return K3MOE_OK;
    }
    K3_TRY(route_into(L, X, xdt, T, st));
    if (L->nev) K3_CUDA(cudaEventRecord(L->ev[1], st));
    if (T == 1 && xdt == K3MOE_F32) {
        ExpertSrc src;
        memset(&src, 0, sizeof(src));
        src.table = L->table;
        src.ids = L->ids;
        K3_TRY(k3::launch_rows_t1(1, (const float *)X, src, L->k, L->d, L->f, L->h, st));
        if (L->nev) K3_CUDA(cudaEventRecord(L->ev[2], st));
        K3_TRY(k3::launch_down_t1(L->h, src, L->w, L->k, L->d, L->f, out, st));
    } else if (L->mxq && L->mxq_ready) {
        int *err = k3::device_error_word();
        K3_TRY(k3::launch_group(L->ids, T * L->k, L->E, k3::grouped_nt(), L->offsets, L->perm,
                                L->items, L->n_items, st));
        K3_TRY(k3::launch_mxq_gateup(X, xdt, T, L->k, L->E, L->d, L->f, L->mx_maps, L->offsets, L->perm,
                                     L->mq_tiles, L->mq_ntiles, L->mq_tbase, L->mq_slot, L->mq_max_tiles,
                                     L->mq_xg, L->mq_xsf, L->mq_hg, L->mq_hsf, err, st));
        if (L->nev) K3_CUDA(cudaEventRecord(L->ev[2], st));
        K3_TRY(k3::launch_mxq_down(T, L->k, L->d, L->f, L->mx_maps, L->perm, L->w, L->mq_tiles, L->mq_ntiles,
                                   L->mq_hg, L->mq_hsf, out, err, st));
    } else if (L->tc && L->tc_ready) {
        int *err = k3::device_error_word();
        K3_TRY(k3::launch_group(L->ids, T * L->k, L->E, k3::grouped_nt(), L->offsets, L->perm,
                                L->items, L->n_items, st));
        const int kd = (L->e4m3 && L->e4m3_ok) ? 1 : 0;
        K3_TRY(k3::launch_tc_gateup(X, xdt, T, kd, L->k, L->E, L->d, L->f, L->table, L->tc_maps, L->offsets,
                                    L->perm, L->tc_tiles, L->tc_ntiles, L->tc_max_tiles, L->tscale, L->Xg,
                                    L->Hg, L->hf, L->hmax, err, st));
        if (L->nev) K3_CUDA(cudaEventRecord(L->ev[2], st));
        K3_TRY(k3::launch_tc_down(T, kd, L->k, L->d, L->f, L->table, L->tc_maps, L->perm, L->w,
                                  L->tc_tiles, L->tc_ntiles, L->Hg, L->hf, L->hmax, out, err, st));
    } else {
        const int npairs = T * L->k;
        K3_TRY(k3::launch_group(L->ids, npairs, L->E, k3::grouped_nt(), L->offsets, L->perm,
                                L->items, L->n_items, st));
        K3_TRY(k3::launch_grouped_gateup(X, xdt, L->table, L->perm, L->items, L->n_items, npairs,
                                         L->k, L->d, L->f, L->h, st));
        if (L->nev) K3_CUDA(cudaEventRecord(L->ev[2], st));
        K3_TRY(k3::launch_grouped_down(L->h, L->table, L->perm, L->items, L->n_items, npairs,
                                       L->k, L->d, L->f, L->w, L->Y, st));
        K3_TRY(k3::launch_combine(L->Y, T, L->k, L->d, out, st));
    }
    if (L->nev) K3_CUDA(cudaEventRecord(L->ev[3], st));
    if (ids_out)
        K3_CUDA(cudaMemcpyAsync(ids_out, L->ids, sizeof(int32_t) * T * L->k,
                                cudaMemcpyDeviceToDevice, st));
    if (w_out)
        K3_CUDA(cudaMemcpyAsync(w_out, L->w, sizeof(float) * T * L->k, cudaMemcpyDeviceToDevice,
                                st));
    return K3MOE_OK;
}

int k3moe_layer_set_option(k3moe_layer *L, int32_t option, int32_t value)
{
    if (!L || (value != 0 && value != 1)) return K3MOE_EINVAL;
    if (option == K3MOE_OPT_FUSED_T1) {
        L->fused = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_ACT_F16) {
        L->act16 = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_TC) {
        L->tc = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_TC_E4M3) {
        L->e4m3 = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_MX) {
        L->mx = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_SIGMOID_ROUTER) {
        L->sigmoid = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_SIGMOID_NORM) {
        L->sig_norm = value != 0;
        return K3MOE_OK;
    }
    if (option == K3MOE_OPT_MXQ) {
        L->mxq = value != 0;
        return K3MOE_OK;
    }
    return K3MOE_EINVAL;
}

int k3moe_layer_fused_t1(const k3moe_layer *L)
{
    if (!L) return K3MOE_EINVAL;
    if (L->mx && L->mx_ready) return 0;  // the block-scaled path takes precedence
    return (L->fused && !L->router_only && k3::fused_t1_supported(L->E, L->k, L->d, L->f)) ? 1 : 0;
}

int k3moe_layer_mx_t1(const k3moe_layer *L)
{
    if (!L) return K3MOE_EINVAL;
    return (L->mx && L->mx_ready) ? 1 : 0;
}

int64_t k3moe_shared_expert_bytes(int32_t d, int32_t f)
{
    if (d <= 0 || f <= 0 || d % 8 || f % 8) return -1;
    return 6 * (int64_t)d * f;
}

int k3moe_shared_expert_view(k3moe_bf16_expert *out, const void *blob, int32_t d, int32_t f)
{
    if (!out || !blob || k3moe_shared_expert_bytes(d, f) < 0 || !aligned16(blob)) return K3MOE_EINVAL;
    const uint16_t *b = (const uint16_t *)blob;
    out->gate = b;
    out->up = b + (size_t)d * f;
    out->down = b + 2 * (size_t)d * f;
    return K3MOE_OK;
}

size_t k3moe_shared_workspace(int32_t n, int32_t f)
{
    if (n <= 0 || n > K3MOE_MAX_SHARED || f <= 0) return 0;
    return sizeof(float) * k3::shared_workspace_floats(n, f);
}

int k3moe_shared_forward(float *out, const float *x, int32_t T, const k3moe_bf16_expert *ex, int32_t n,
                         int32_t d, int32_t f, int32_t accumulate, void *ws, size_t ws_bytes, k3moe_stream s)
{
    if (!out || !x || !ex || !ws || T <= 0 || n <= 0 || n > K3MOE_MAX_SHARED || !k3::shared_supported(n, d, f) ||
        !aligned16(out) || !aligned16(x) || !aligned16(ws) || ws_bytes < k3moe_shared_workspace(n, f))
        return K3MOE_EINVAL;
    const uint16_t *g[K3MOE_MAX_SHARED], *u[K3MOE_MAX_SHARED], *dn[K3MOE_MAX_SHARED];
    for (int i = 0; i < n; i++) {
        if (!ex[i].gate || !ex[i].up || !ex[i].down || !aligned16(ex[i].gate) || !aligned16(ex[i].up) ||
            !aligned16(ex[i].down))
            return K3MOE_EINVAL;
        g[i] = ex[i].gate;
        u[i] = ex[i].up;
        dn[i] = ex[i].down;
    }
    return k3::launch_shared(g, u, dn, n, x, T, d, f, (float *)ws, out, accumulate ? 1 : 0, cs(s));
}

int k3moe_layer_mxq(const k3moe_layer *L)
{
    if (!L) return K3MOE_EINVAL;
    return (L->mxq && L->mxq_ready) ? 1 : 0;
}

int k3moe_mx_quantize(uint8_t *codes, uint8_t *scales, const void *x, int x_dtype, int32_t rows, int32_t cols,
                      k3moe_stream s)
{
    if (!codes || !scales || !x || rows <= 0 || cols <= 0 || cols % 32 ||
        (x_dtype != K3MOE_F32 && x_dtype != K3MOE_BF16))
        return K3MOE_EINVAL;
    return k3::launch_mx_quantize(x, x_dtype, rows, cols, codes, scales, cs(s));
}

int k3moe_layer_set_events(k3moe_layer *L, void *const *host_events, int32_t n)
{
    if (!L || n < 0 || (n > 0 && (n < 4 || !host_events))) return K3MOE_EINVAL;
    L->nev = n ? 4 : 0;
    for (int i = 0; i < L->nev; i++) {
        if (!host_events[i]) {
            L->nev = 0;
            return K3MOE_EINVAL;
        }
        L->ev[i] = (cudaEvent_t)host_events[i];
    }
    return K3MOE_OK;
}

int k3moe_layer_experts_t1(k3moe_layer *L, const float *x, const k3moe_expert *sel,
                           const float *w, int32_t k, float *out, k3moe_stream s)
{
    if (!L || !x || !sel || !w || !out || k < 1 || k > k3::kMaxInline || k > L->k)
        return K3MOE_EINVAL;
    if (!aligned16(x) || !aligned16(out)) return K3MOE_EINVAL;
    ExpertSrc src;
    memset(&src, 0, sizeof(src));
    for (int j = 0; j < k; j++) {
        if (!valid_expert(sel[j], L->d, L->f)) return K3MOE_EINVAL;
        src.inl[j] = to_dev(sel[j]);
    }
    K3_TRY(k3::launch_rows_t1(1, x, src, k, L->d, L->f, L->h, cs(s)));
    return k3::launch_down_t1(L->h, src, w, k, L->d, L->f, out, cs(s));
}

int k3moe_rmsnorm(float *u, const float *x, int32_t n, float eps, k3moe_stream s)
{
    if (!u || !x || n <= 0 || !(eps >= 0.f)) return K3MOE_EINVAL;
    return k3::launch_rmsnorm(u, x, n, eps, cs(s));
}

int k3moe_residual_add(float *x, const float *delta, int32_t n, k3moe_stream s)
{
    if (!x || !delta || n <= 0) return K3MOE_EINVAL;
    return k3::launch_residual(x, delta, n, cs(s));
}

}  // extern "C"

// ------------------------------------------------------ streamed decode loop

extern "C" int k3moe_stream_decode(const k3moe_stream_desc *D, const float *X, int32_t T,
                                   float *out, int32_t *host_ids_out, uint8_t *host_hit_out,
                                   k3moe_stream s)
{
    if (!D || !D->host_layers || !D->cache || D->n_layers <= 0 || !X || !out || T <= 0 ||
        !(D->eps >= 0.f) || !aligned16(X) || !aligned16(out))
        return K3MOE_EINVAL;
    const k3moe_layer *L0 = D->host_layers[0];
    if (!L0) return K3MOE_EINVAL;
    const int E = L0->E, k = L0->k, d = L0->d, f = L0->f;
    if (k > k3::kMaxInline) return K3MOE_EINVAL;
    const int nsh = D->trunk ? D->n_shared : 0;
    if (D->trunk && (nsh <= 0 || nsh > K3MOE_MAX_SHARED || !k3::shared_supported(nsh, d, f))) return K3MOE_EINVAL;
    for (int l = 0; l < D->n_layers; l++) {
        const k3moe_layer *L = D->host_layers[l];
        if (!L || L->E != E || L->k != k || L->d != d || L->f != f) return K3MOE_EINVAL;
    }
    cudaStream_t st = cs(s);
    float *xcur = nullptr, *u = nullptr, *wsub = nullptr, *shws = nullptr;
    float *whost = nullptr;  // pinned: [k] routing weights, then [k] reordered hits-first
    int32_t *idhost = nullptr;
    int rc = K3MOE_OK;
    auto fail = [&](int code) {
        if (rc == K3MOE_OK) rc = code;
    };
    if (cudaMalloc(&xcur, sizeof(float) * d) != cudaSuccess ||
        cudaMalloc(&u, sizeof(float) * d) != cudaSuccess ||
        cudaMalloc(&wsub, sizeof(float) * k) != cudaSuccess ||
        cudaMallocHost(&idhost, sizeof(int32_t) * k) != cudaSuccess ||
        cudaMallocHost(&whost, sizeof(float) * 2 * k) != cudaSuccess ||
        (nsh && cudaMalloc(&shws, k3moe_shared_workspace(nsh, f)) != cudaSuccess)) {
        cudaGetLastError();
        fail(K3MOE_ENOMEM);
    }
    std::vector<int64_t> keys(k);
    std::vector<void *> blobs(k);
    std::vector<uint8_t> hits(k);
    std::vector<int> order(k);
    for (int t = 0; t < T && rc == K3MOE_OK; t++) {
        if (cudaMemcpyAsync(xcur, X + (size_t)t * d, sizeof(float) * d, cudaMemcpyDeviceToDevice,
                            st) != cudaSuccess) {
            fail(K3MOE_ECUDA);
            break;
        }
        for (int l = 0; l < D->n_layers && rc == K3MOE_OK; l++) {
            k3moe_layer *L = D->host_layers[l];
            // RMSNorm folded into the router: u = x / sqrt(mean(x^2) + eps)
            int r = k3::launch_route_t1(xcur, K3MOE_F32, L->Wr, E, d, L->part, L->logits, router_of(L),
                                        k, L->ids, L->w, L->ticket, D->eps, u, st);
            if (r != K3MOE_OK) {
                fail(r);
                break;
            }
            if (cudaMemcpyAsync(idhost, L->ids, sizeof(int32_t) * k, cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess ||
                cudaMemcpyAsync(whost, L->w, sizeof(float) * k, cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess ||
                cudaStreamSynchronize(st) != cudaSuccess) {
                cudaGetLastError();
                fail(K3MOE_ECUDA);
                break;
            }
            for (int j = 0; j < k; j++) keys[j] = (int64_t)l * E + idhost[j];
            // The misses' copies run on a side stream while the hits are
            // computed; each miss is then computed as soon as its own copy is
            // in, so that only the last miss's compute follows the copies.
            r = k3moe_cache_acquire_split(D->cache, keys.data(), k, blobs.data(), hits.data(), s);
            if (r != K3MOE_OK) {
                fail(r);
                break;
            }
            int nh = 0;
            for (int j = 0; j < k; j++)
                if (hits[j]) order[nh++] = j;
            for (int j = 0, q = nh; j < k; j++)  // misses in key order = copy order
                if (!hits[j]) order[q++] = j;
            ExpertSrc src;
            memset(&src, 0, sizeof(src));
            for (int q = 0; q < k && r == K3MOE_OK; q++) {
                whost[k + q] = whost[order[q]];
                k3moe_expert v;
                r = k3moe_expert_view(&v, blobs[order[q]], d, f);
                if (r == K3MOE_OK) src.inl[q] = to_dev(v);
            }
            // whost[k..] is rewritten only after the next layer's synchronise,
            // when this copy has long completed
            if (r == K3MOE_OK && cudaMemcpyAsync(wsub, whost + k, sizeof(float) * k,
                                                 cudaMemcpyHostToDevice, st) != cudaSuccess)
                r = K3MOE_ECUDA;
            // x += sum_j w_j expert_j(u): the down kernel adds into x
            if (r == K3MOE_OK && nh > 0) {
                r = k3::launch_rows_t1(1, u, src, nh, d, f, L->h, st);
                if (r == K3MOE_OK) r = k3::launch_down_t1(L->h, src, wsub, nh, d, f, xcur, st, true);
            }
            // x += the layer's shared experts, from its trunk bytes (while the
            // misses still copy)
            if (r == K3MOE_OK && nsh) {
                void *tb = nullptr;
                r = k3moe_trunk_acquire(D->trunk, l, &tb, nullptr, s);
                const uint16_t *g[K3MOE_MAX_SHARED], *uu[K3MOE_MAX_SHARED], *dn[K3MOE_MAX_SHARED];
                for (int q = 0; q < nsh && r == K3MOE_OK; q++) {
                    k3moe_bf16_expert se;
                    r = k3moe_shared_expert_view(&se, (const uint8_t *)tb + (size_t)q * k3moe_shared_expert_bytes(d, f),
                                                 d, f);
                    g[q] = se.gate;
                    uu[q] = se.up;
                    dn[q] = se.down;
                }
                if (r == K3MOE_OK) r = k3::launch_shared(g, uu, dn, nsh, u, 1, d, f, shws, xcur, 1, st);
                if (tb) {
                    const int rt = k3moe_trunk_release(D->trunk, l, s);
                    if (r == K3MOE_OK) r = rt;
                }
            }
            for (int q = nh; q < k && r == K3MOE_OK; q++) {
                r = k3moe_cache_wait_copy(D->cache, blobs[order[q]], s);
                ExpertSrc one;
                memset(&one, 0, sizeof(one));
                one.inl[0] = src.inl[q];
                if (r == K3MOE_OK) r = k3::launch_rows_t1(1, u, one, 1, d, f, L->h, st);
                if (r == K3MOE_OK) r = k3::launch_down_t1(L->h, one, wsub + q, 1, d, f, xcur, st, true);
            }
            const int rr = k3moe_cache_release(D->cache, s);
            if (r == K3MOE_OK) r = rr;
            if (r != K3MOE_OK) {
                fail(r);
                break;
            }
            const size_t o = ((size_t)t * D->n_layers + l) * k;
            if (host_ids_out) memcpy(host_ids_out + o, idhost, sizeof(int32_t) * k);
            if (host_hit_out) memcpy(host_hit_out + o, hits.data(), k);
        }
        if (rc == K3MOE_OK &&
            cudaMemcpyAsync(out + (size_t)t * d, xcur, sizeof(float) * d, cudaMemcpyDeviceToDevice,
                            st) != cudaSuccess)
            fail(K3MOE_ECUDA);
    }
    cudaStreamSynchronize(st);
    cudaGetLastError();
    cudaFree(xcur);
    cudaFree(u);
    cudaFree(wsub);
    if (shws) cudaFree(shws);
    cudaFreeHost(idhost);
    cudaFreeHost(whost);
    return rc;
}
