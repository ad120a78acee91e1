/*
 * k3moe.h -- C ABI of the GB300 (sm_103a) MXFP4 routed-expert MoE library.
 *
 * The library computes the routed-expert layer of a mixture-of-experts
 * decoder straight from packed MXFP4 weights: router logits, top-k selection
 * with combine weights from the unbiased scores, and for every selected
 * expert the gate/up products, SwiGLU, the down product and the weighted
 * combine.  The 4-bit codes feed block-scaled tensor-core products as stored
 * (batch 1) or are decoded on chip, in registers or shared memory; no weight
 * is ever expanded in device memory.
 *
 * Sources of the operations (page title, section):
 *  [EXPL]  "kimi-k3-in-c" explainer, ai.thesatyajit.com
 *  [ENG]   "kimi-k3-in-c: A 176 KB Engine That Runs a 2.78T-Parameter MoE in
 *          8 GB of RAM", aniketkarneai.com
 *  [LOCAL] "Running Kimi K3 locally: activation sparsity as architecture",
 *          zorost.com
 *  [HOW]   "How kimi-k3-in-c Runs a 2.8-Trillion-Parameter Model on 8 GB of
 *          RAM", dimitriaigle.fr
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers unless the parameter name starts with
 *    `host_`.  Device buffers must be 16-byte aligned.
 *  - The caller owns every buffer it passes; the library owns only the objects
 *    it creates (layer, cache, trunk) and frees them in the matching destroy
 *    call.
 *  - Work is enqueued on the caller's stream `s` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns before the GPU finishes.  Outputs are
 *    valid once the stream has reached that point.
 *  - Every call returns a status: K3MOE_OK (0) or a negative K3MOE_E* code.
 *    Invalid arguments are refused with K3MOE_EINVAL before anything is
 *    enqueued; nothing is guessed or defaulted (a zero or inconsistent size is
 *    an error).  No call exits the process or throws.
 *  - A NaN E8M0 scale (byte 255) is not an error: its 32-group contributes 0
 *    [ENG, "What byte-identical actually costs"].
 *  - Device kernels never trap.  Errors detected on the device (a bounded
 *    wait that ran out) are recorded in a device error word that
 *    k3moe_device_error() reads and clears.  The word is a file-scope device
 *    variable (one int per device, zero at load), so no path allocates for
 *    it; every entry point, k3moe_expert_gemv_noalloc included, reports
 *    through it.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */

#define K3MOE_OK        0
#define K3MOE_EINVAL   (-1)  /* bad argument: size, alignment, null pointer   */
#define K3MOE_ENOMEM   (-2)  /* an allocation the call needs failed           */
#define K3MOE_ECUDA    (-3)  /* a CUDA runtime call failed                    */
#define K3MOE_ETIMEOUT (-4)  /* a bounded device or host wait ran out          */
#define K3MOE_EBUSY    (-5)  /* cache or trunk: no free slot for the request  */
#define K3MOE_ENODEV   (-6)  /* no usable sm_103 device                       */
#define K3MOE_EIO      (-7)  /* a file could not be opened, read or written   */

/* Input activation types for k3moe_layer_forward. */
#define K3MOE_F32  0
#define K3MOE_BF16 1

typedef struct CUstream_st *k3moe_stream; /* same object as cudaStream_t */

/* Human-readable name of a status code (static string). */
const char *k3moe_strerror(int status);

/* Library ABI version, (major << 16) | minor. */
int k3moe_version(void);

/* Reads and clears the device error word of the current device
 * (0 = none, else a K3MOE_E* code).  Synchronises the device. */
int k3moe_device_error(void);

/* Self-check of the bounded waits (the pages have no counterpart; every
 * wait in this library's kernels is bounded so that a lost producer ends in
 * an error status instead of a hung GPU).  Enqueues one CTA that waits on a
 * barrier nothing completes; after the 2 s limit it records K3MOE_ETIMEOUT
 * in the device error word and exits normally.  Returns K3MOE_OK when the
 * launch was enqueued; read the outcome with k3moe_device_error(). */
int k3moe_check_wait_timeout(k3moe_stream s);

/* ---------------------------------------------------------- packed format */

/*
 * One MXFP4 matrix W[rows][in] in the pages' canonical layout [EXPL,
 * "Reduction one: the experts already ship at half a byte"]:
 *   packed : [rows][in/2] bytes, two 4-bit E2M1 codes per byte; the LOW nibble
 *            holds the even-index weight, the high nibble the odd one [LOCAL,
 *            "What are the four reductions, and why is the answer unchanged?"]
 *   scales : [rows][in/32] bytes, one E8M0 exponent e per 32 consecutive
 *            weights of a row; value = E2M1(code) * 2^(e-127); e = 255 zeroes
 *            the group.
 * 0.53125 bytes per weight [ENG, "The four reductions"].  `in` must be a
 * multiple of 32.  Both planes must be 16-byte aligned.
 */
typedef struct {
    const uint8_t *packed;
    const uint8_t *scales;
    int32_t rows;
    int32_t in;
} k3moe_mat;

/* One routed expert: gate and up are [f x d], down is [d x f]. */
typedef struct {
    k3moe_mat gate;
    k3moe_mat up;
    k3moe_mat down;
} k3moe_expert;

/* Packed bytes of a rows x in matrix: rows * (in/2 + in/32); -1 if invalid. */
int64_t k3moe_matrix_bytes(int32_t rows, int32_t in);

/* Packed bytes of one expert, 3 matrices; 17,547,264 for d=7168, f=1536
 * [ENG, "The four reductions"; EXPL, "Reduction one"].  -1 if invalid. */
int64_t k3moe_expert_bytes(int32_t d, int32_t f);

/*
 * HBM layout of one expert: a single blob of k3moe_expert_bytes(d, f) bytes
 * holding, in order, gate.packed, gate.scales, up.packed, up.scales,
 * down.packed, down.scales (every plane size is a multiple of 16 bytes for
 * d, f multiples of 32).  k3moe_expert_view fills *out with the six plane
 * pointers inside `blob` (pure host arithmetic, no CUDA call).
 */
int k3moe_expert_view(k3moe_expert *host_out, const void *blob, int32_t d, int32_t f);

/*
 * Packs the six canonical planes (each in host or device memory) into one
 * expert blob (device memory, caller-owned, k3moe_expert_bytes(d, f) bytes),
 * by stream-ordered copies on `s`.  Plane shapes as in k3moe_mat.
 */
int k3moe_pack_expert(void *blob, const uint8_t *gate_packed, const uint8_t *gate_scales,
                      const uint8_t *up_packed, const uint8_t *up_scales,
                      const uint8_t *down_packed, const uint8_t *down_scales, int32_t d,
                      int32_t f, k3moe_stream s);

/* ------------------------------------------------------ expert products */

/*
 * y[rows] = W x for one packed matrix: the pages' primitive
 * k3_matmul_mxfp4 [EXPL, "Reduction one"], here with fp32 accumulation.
 * x: fp32 [W->in]; y: fp32 [W->rows]. `host_W` is a host struct holding
 * device plane pointers.
 */
int k3moe_matmul_mxfp4(float *y, const float *x, const k3moe_mat *host_W, k3moe_stream s);

/*
 * One expert, one token: y = W_down (silu(W_gate x) * (W_up x)),
 * silu(z) = z / (1 + e^-z).  x fp32 [d], y fp32 [d].
 * `workspace` is caller-owned device scratch of at least
 * k3moe_expert_gemv_workspace(d, f) bytes (it holds the SwiGLU output h).
 */
size_t k3moe_expert_gemv_workspace(int32_t d, int32_t f);
int k3moe_expert_gemv(float *y, const float *x, const k3moe_expert *host_e, int32_t d,
                      int32_t f, void *workspace, size_t workspace_bytes, k3moe_stream s);

/*
 * k3moe_expert_gemv without a workspace, for callers that cannot allocate
 * device memory on the call path: code running while a stream is captured in
 * global capture mode, threads with a no-allocation rule, plug-ins that must
 * not touch the host application's allocator, systems that budget device
 * memory once at start-up.  (The pages have no counterpart; this is a
 * deployment convenience of this library.)
 *  - Same arguments, layout and result as k3moe_expert_gemv, minus the
 *    workspace; the SwiGLU intermediate lives in a file-scope device array of
 *    K3MOE_NOALLOC_MAX_F floats held by every device that loads the library
 *    until the process exits.  f > K3MOE_NOALLOC_MAX_F is refused with
 *    K3MOE_EINVAL.
 *  - Allocates nothing: no cudaMalloc/cudaFree or allocating library call.
 *  - The first call on a device (with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - A bounded wait that runs out in its kernels is recorded in the device
 *    error word: the call itself returns K3MOE_OK once the kernels are
 *    enqueued; read the outcome with k3moe_device_error().
 *  - All calls on a device share the array: calls whose kernels overlap on the
 *    GPU race, so serialise them.  Each call overwrites the array fully before
 *    reading it.
 */
#define K3MOE_NOALLOC_MAX_F 2048
int k3moe_expert_gemv_noalloc(float *y, const float *x, const k3moe_expert *host_e, int32_t d,
                              int32_t f, k3moe_stream s);

/*
 * MXFP4 quantisation of activations (the conversion K3MOE_OPT_MXQ applies;
 * the pages quantise only the weights, so the rule is the OCP Microscaling
 * v1.0 conversion to E2M1 with one E8M0 scale per 32): per 32-block of a row
 * the scale byte is e = floor(log2 amax) - 2 + 127 clamped to [0, 254] (the
 * block's largest magnitude amax; e = 0 for an all-zero block); each value
 * divided by 2^(e-127) rounds to the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6,
 * ties to the even code, larger magnitudes saturating to 6; the sign is bit
 * 3 of the code (a negative value that rounds to 0 gives code 8).  A block
 * holding a non-finite value gets scale byte 255 and codes 0.
 *  x       device, [rows][cols], x_dtype K3MOE_F32 or K3MOE_BF16, cols a
 *          multiple of 32
 *  codes   device, [rows][cols/2] bytes (out): two codes per byte, the even
 *          element in the low nibble (the weights' packing)
 *  scales  device, [rows][cols/32] bytes (out)
 * Errors: K3MOE_EINVAL for null pointers, sizes <= 0, cols % 32 != 0.
 */
int k3moe_mx_quantize(uint8_t *codes, uint8_t *scales, const void *x, int x_dtype, int32_t rows,
                      int32_t cols, k3moe_stream s);

/* ----------------------------------------------------------------- layer */

/*
 * A routed-expert MoE layer with all experts resident in HBM.
 *  n_experts  E (896 on the pages [ENG, intro]), top_k (16)
 *  d, f       hidden and expert intermediate sizes (multiples of 32)
 *  router_w   bf16 [E x d] row-major (the router is part of the bf16 trunk)
 *  sel_bias   fp32 [E] added to the logits for SELECTION only, or NULL.  The
 *             combine weights always come from the unbiased logits [LOCAL,
 *             "How is the C engine actually built?", invariant 3].
 *  host_experts  host array of E expert views (device plane pointers); the
 *             table is copied at create, the weights are not.  NULL makes a
 *             router-only layer (route and experts_t1 only, for experts that
 *             live in an expert cache).
 *  max_tokens the largest T that forward will be called with (sizes the
 *             library-owned scratch).
 * Returns K3MOE_EINVAL on any zero/invalid field, K3MOE_ENOMEM if the scratch
 * cannot be allocated.
 */
typedef struct {
    int32_t n_experts;
    int32_t top_k;
    int32_t d;
    int32_t f;
    const uint16_t *router_w;
    const float *sel_bias;
    const k3moe_expert *host_experts;
    int32_t max_tokens;
} k3moe_layer_desc;

typedef struct k3moe_layer k3moe_layer;

int k3moe_layer_create(k3moe_layer **host_out, const k3moe_layer_desc *host_desc);
int k3moe_layer_destroy(k3moe_layer *L);

/*
 * Routing only: logits = X W_r^T (fp32 accumulation), the top_k experts by
 * logit + sel_bias (ties to the lower id), ids ascending, and w = softmax of
 * the unbiased logits over the chosen set (or the sigmoid rule of
 * K3MOE_OPT_SIGMOID_ROUTER below).
 *  X    [T x d], x_dtype K3MOE_F32 or K3MOE_BF16
 *  ids  int32 [T x top_k] (out), w fp32 [T x top_k] (out)
 */
int k3moe_layer_route(k3moe_layer *L, const void *X, int x_dtype, int32_t T, int32_t *ids,
                      float *w, k3moe_stream s);

/*
 * The whole layer: out[t] = sum_j w[t][j] * expert_{ids[t][j]}(X[t]).
 *  X    [T x d] (x_dtype), out fp32 [T x d]
 *  ids_out / w_out  optional (NULL allowed) copies of the routing result.
 * 1 <= T <= max_tokens.  T = 1 runs the fused batch-1 path; T > 1 groups the
 * (token, slot) pairs by expert and runs grouped products.
 */
int k3moe_layer_forward(k3moe_layer *L, const void *X, int x_dtype, int32_t T, float *out,
                        int32_t *ids_out, float *w_out, k3moe_stream s);

/*
 * Layer options (value 0/1):
 *  K3MOE_OPT_FUSED_T1  batch-1 fp32 forward runs as one persistent
 *                      cooperative kernel (router, top-k, experts, combine)
 *                      when the shape allows it (d % 1024 == 0, d <= 7168,
 *                      f % 512 == 0, f <= 2048); default 1.  0 selects the
 *                      three-kernel path.
 *  K3MOE_OPT_ACT_F16   on the fused batch-1 path, round the activations of
 *                      the expert products to f16 (11 significant bits, one
 *                      power-of-two scale per 16 activations) and use one
 *                      fp32-accumulating FMA per weight; default 0, which
 *                      keeps each activation as an exact f16 hi + lo pair
 *                      (two FMAs per weight, fp32-class products).  The
 *                      rounding adds a relative error of order 2^-12 per
 *                      activation; the router is fp32 either way.
 *  K3MOE_OPT_TC        multi-token forwards (and bf16 batch-1 forwards) of a
 *                      layer created with max_tokens > 1 run the expert
 *                      products as grouped tcgen05 MMAs: weights decoded
 *                      exactly to bf16 in shared memory, fp32 activations and
 *                      the SwiGLU output split into bf16 hi + lo (16
 *                      significant bits), fp32 accumulation, the weighted
 *                      combine by fp32 atomic adds (summation order not
 *                      fixed).  Needs d % 256 == 0 and f % 256 == 0; default 1.
 *                      0 selects the CUDA-core grouped path.
 *  K3MOE_OPT_TC_E4M3   on the K3MOE_OPT_TC path, run the expert products
 *                      with e4m3 operands (kind::f8f6f4): weights decoded
 *                      exactly to e4m3 (possible when every scale byte of
 *                      the layer is in [119, 133] or 255, checked at layer
 *                      creation; otherwise the option has no effect),
 *                      activations and h as e4m3 pieces with power-of-two
 *                      scales (4 pieces for fp32 tokens and for h, each
 *                      element then within 2^-15 of its token's or pair's
 *                      largest magnitude; 2 for bf16 tokens, exact but for
 *                      elements below about 2^-10 of that magnitude).
 *                      Default 1.
 *  K3MOE_OPT_MX        batch-1 forwards of a layer with a resident expert
 *                      table run the expert products on the block-scaled
 *                      tensor cores (tcgen05.mma kind::mxf4): the packed
 *                      E2M1 planes and their E8M0 scales are the A operand
 *                      as stored, with no decode; the activations (and h)
 *                      are the B operand as 16 E2M1 pieces per 32-block
 *                      with one E8M0 scale each, exact in fp32 to below
 *                      2e-8 of the block's largest magnitude; fp32
 *                      accumulation; the weighted combine by fp32
 *                      reductions (summation order not fixed).
 *                      Needs d % 512 == 0, f % 512 == 0, d <= 8192,
 *                      f <= 2048, top_k <= 16.  Takes precedence over
 *                      K3MOE_OPT_FUSED_T1.  Default 1.
 *  K3MOE_OPT_SIGMOID_ROUTER  the router scores each expert with
 *                      s = 1 / (1 + e^-logit), selects the top_k largest
 *                      s + sel_bias and weights the chosen experts with their
 *                      UNBIASED scores s ("Running Kimi K3 locally", "How is
 *                      the C engine actually built?", invariant 3).  Default
 *                      0: selection on logit + sel_bias, weights the softmax
 *                      of the chosen logits.  Applies to every path.
 *  K3MOE_OPT_SIGMOID_NORM  with K3MOE_OPT_SIGMOID_ROUTER, the weights are
 *                      divided by their sum over the chosen set (the pages do
 *                      not say whether they are renormalised).  Default 0.
 *  K3MOE_OPT_MXQ       multi-token forwards (T > 1) of a layer created with
 *                      max_tokens > 1 quantise the activations to MXFP4 and
 *                      run the expert products as block-scaled E2M1 x E2M1
 *                      GEMMs (tcgen05.mma kind::mxf4, weights as stored): x
 *                      per 32-block along d and h = silu(g) * u (held in
 *                      fp32) per 32-block along f, each by the conversion of
 *                      k3moe_mx_quantize; fp32 accumulation; the weighted
 *                      combine by fp32 reductions.  The pages quantise only
 *                      the weights this way ["kimi-k3-in-c" explainer,
 *                      "Reduction one"]; quantising the activations too is a
 *                      different contract: the result is the layer of
 *                      quantised activations (about 10% from the exact one
 *                      per output vector), not the exact layer.  Needs
 *                      d % 512 == 0, f % 512 == 0.  Default 0.
 * k3moe_layer_fused_t1 returns 1 when a batch-1 fp32 forward of this layer
 * would run fused (the block-scaled path is off or unsupported), else 0
 * (negative on error).  After a device-side timeout
 * (k3moe_device_error() == K3MOE_ETIMEOUT) a layer must be recreated.
 */
#define K3MOE_OPT_FUSED_T1 1
#define K3MOE_OPT_ACT_F16  2
#define K3MOE_OPT_TC       4
#define K3MOE_OPT_TC_E4M3  8
#define K3MOE_OPT_MX       16
#define K3MOE_OPT_SIGMOID_ROUTER 32
#define K3MOE_OPT_SIGMOID_NORM   64
#define K3MOE_OPT_MXQ            128
int k3moe_layer_set_option(k3moe_layer *L, int32_t option, int32_t value);
int k3moe_layer_fused_t1(const k3moe_layer *L);
/* 1 when a batch-1 forward of this layer runs on the block-scaled tensor
 * cores (K3MOE_OPT_MX set and the layer supports it), else 0. */
int k3moe_layer_mx_t1(const k3moe_layer *L);
/* 1 when a multi-token forward of this layer runs with MXFP4 activations
 * (K3MOE_OPT_MXQ set and the layer has its buffers and tensor maps), else 0. */
int k3moe_layer_mxq(const k3moe_layer *L);

/*
 * Timing hook: when set, every later k3moe_layer_forward records
 * host_events[0] on its stream before the first kernel, [1] after routing,
 * [2] after the gate/up products and [3] after the down products and combine
 * (cudaEvent_t handles, created and owned by the caller).  n = 0 clears it.
 * On the fused batch-1 path the whole layer is one kernel: [1] and [2] are
 * recorded together with [3] after it.
 */
int k3moe_layer_set_events(k3moe_layer *L, void *const *host_events, int32_t n);

/*
 * Batch-1 experts for an explicit expert list, e.g. slots handed out by the
 * expert cache: out = sum_j w[j] * expert_j(x) over host_sel[0..k).
 *  host_sel  host array of k expert views (device pointers), k <= 16
 *  w         fp32 [k] combine weights (device)
 *  x         fp32 [d], out fp32 [d]
 */
int k3moe_layer_experts_t1(k3moe_layer *L, const float *x, const k3moe_expert *host_sel,
                           const float *w, int32_t k, float *out, k3moe_stream s);

/*
 * RMSNorm with residual, as used between streamed layers:
 *  u = x / sqrt(mean(x^2) + eps)   (epsilon inside the square root [ENG,
 *  "What byte-identical actually costs"]; unit gain).  x fp32 [n], u fp32 [n].
 */
int k3moe_rmsnorm(float *u, const float *x, int32_t n, float eps, k3moe_stream s);

/* x += delta, fp32 [n]. */
int k3moe_residual_add(float *x, const float *delta, int32_t n, k3moe_stream s);

/* ------------------------------------------------------------ expert cache */

/*
 * HBM-resident LRU cache of expert blobs fed from pinned host memory
 * [EXPL, "The cache the project exists for", "The bug the code confesses
 * to"; HOW, "The LRU cache: which experts to keep hot"].
 *
 * Keys are (layer * n_experts + expert).  The arena holds
 * floor(capacity_bytes / expert_bytes) slots.  Each slot is EMPTY, INFLIGHT
 * (reserved by a batch whose copy has not been waited for) or holds a key.
 * A batch acquire first marks its hits, then gives every miss a DISTINCT slot
 * (an EMPTY one, else the least recently used slot that is neither pinned nor
 * used by the same batch), marks it INFLIGHT, and issues one host->HBM copy of
 * expert_bytes per miss on a library-owned side stream; the caller's
 * `compute` stream is made to wait for those copies (events), so kernels
 * enqueued on it afterwards see the data.
 *
 *  host_blobs  host array of n_layers * n_experts pointers to each expert's
 *              blob in host memory (pinned by the caller for full speed).
 * create returns K3MOE_ENOMEM if the arena cannot be allocated (it refuses
 * up front instead of failing later), K3MOE_EINVAL if it holds < 1 slot.
 */
typedef struct k3moe_cache k3moe_cache;

typedef struct {
    int64_t lookups;
    int64_t hits;
    int64_t misses;
    int64_t evictions;
    int64_t h2d_bytes;  /* bytes copied host -> HBM for misses            */
    int64_t hbm_bytes;  /* expert bytes handed to kernels (hits + misses) */
    int32_t slots;
    int32_t pinned;
    int32_t inflight;
    int32_t reserved;
} k3moe_cache_stats;

int k3moe_cache_create(k3moe_cache **host_out, size_t capacity_bytes, size_t expert_bytes,
                       const void *const *host_blobs, int32_t n_layers, int32_t n_experts);
int k3moe_cache_destroy(k3moe_cache *C);

/*
 * Resolves n keys (host array) to device blob pointers (host_blobs_out[n]).
 * host_hit_out (optional) receives 1 per hit, 0 per miss.  Returns
 * K3MOE_EBUSY if a miss finds no evictable slot (nothing is changed then).
 */
int k3moe_cache_acquire(k3moe_cache *C, const int64_t *host_keys, int32_t n,
                        void **host_blobs_out, uint8_t *host_hit_out, k3moe_stream compute);

/*
 * Split form of k3moe_cache_acquire, so that the hits can be computed while
 * the misses copy: the same plan, the same copies and the same outputs, but
 * `compute` is NOT made to wait for the copies and the misses' slots stay
 * INFLIGHT.  Hit pointers may be used on `compute` at once; miss pointers
 * only after k3moe_cache_wait_copies(C, compute).  A later acquire (either
 * form) and k3moe_cache_release wait for the pending copies themselves first.
 */
int k3moe_cache_acquire_split(k3moe_cache *C, const int64_t *host_keys, int32_t n,
                              void **host_blobs_out, uint8_t *host_hit_out,
                              k3moe_stream compute);

/* Makes `compute` wait for every copy issued by an acquire and not yet waited
 * for, and publishes those keys.  Returns the copier's code of the first
 * failed wait (that slot becomes EMPTY and its key uncached). */
int k3moe_cache_wait_copies(k3moe_cache *C, k3moe_stream compute);

/* The same for one blob pointer handed out by an acquire: `compute` waits
 * for that slot's copy only (no-op for a hit or a copy already waited for).
 * The copies of one acquire land in the order of their keys, so a caller can
 * compute on the first misses while the later ones are still copying.
 * K3MOE_EINVAL if blob is not a slot of this cache. */
int k3moe_cache_wait_copy(k3moe_cache *C, const void *blob, k3moe_stream compute);

/* Ends the use of every slot handed out since the previous release: records
 * on `compute` the point after which those slots may be overwritten (a later
 * miss that evicts one of them makes its copy wait for that point).  Slots
 * acquired and not yet released are never evicted. */
int k3moe_cache_release(k3moe_cache *C, k3moe_stream compute);

/* Pins a key: it is loaded if absent (stream-ordered on `compute`) and never
 * evicted afterwards.  K3MOE_EBUSY if no slot can hold it. */
int k3moe_cache_pin(k3moe_cache *C, int64_t key, k3moe_stream compute);

int k3moe_cache_get_stats(k3moe_cache *C, k3moe_cache_stats *host_out);

/* Request histogram: n_layers * n_experts counters of how often each key was
 * asked for [EXPL, "The cache the project exists for"].  Host memory owned
 * by the cache; valid until destroy. */
const uint32_t *k3moe_cache_histogram(const k3moe_cache *C);

/*
 * Copier interface, for tests of the host logic without a GPU: the cache
 * calls alloc_arena once at create, copy() per miss (after the slot's last
 * release), wait() before handing a copied slot's pointer out, release() per
 * slot in k3moe_cache_release, and free_arena at destroy.  Return 0 on
 * success, a negative K3MOE_E* code on failure.  A failed copy leaves its slot
 * EMPTY and the key uncached, and acquire returns the copier's code.  A cache
 * created with a copier makes no CUDA call; its `compute` arguments are
 * passed through untouched.
 */
typedef struct {
    void *ctx;
    int (*alloc_arena)(void *ctx, size_t bytes, void **arena_out);
    int (*free_arena)(void *ctx, void *arena);
    int (*copy)(void *ctx, int32_t slot, void *dst, const void *src, size_t bytes);
    int (*wait)(void *ctx, int32_t slot);
    int (*release)(void *ctx, int32_t slot);
} k3moe_copier;

int k3moe_cache_create_with_copier(k3moe_cache **host_out, size_t capacity_bytes,
                                   size_t expert_bytes, const void *const *host_blobs,
                                   int32_t n_layers, int32_t n_experts,
                                   const k3moe_copier *host_copier);

/* Slot index that holds `key`, or -1 (for tests). */
int32_t k3moe_cache_slot_of(const k3moe_cache *C, int64_t key);

/* ------------------------------------------------- cache policy tooling */

/*
 * Tools for choosing what the cache keeps: the pages keep a request
 * histogram so that a hot set can be measured and pinned rather than
 * guessed [EXPL, "The cache the project exists for"], size the expert cache
 * from a recorded trace replayed offline [LOCAL, "the four reductions"], and
 * compare LRU with Belady's offline optimum over capacities [ENG, "The
 * interesting design decisions"].  All host-side: no CUDA call.
 *
 * A trace is n_batches batches of keys (one batch = the keys one acquire
 * asked for, e.g. one token's experts at one layer): batch_len[b] >= 1 keys
 * each, concatenated in keys[] (sum of batch_len keys, each >= 0).
 */
#define K3MOE_POLICY_LRU    0  /* the live cache's policy, decision for decision  */
#define K3MOE_POLICY_BELADY 1  /* offline optimum: evict the farthest next use    */

/* Starts (on != 0; the record is cleared) or stops recording the keys of
 * every acquire that is placed (a refused batch is not recorded; pins are
 * not requests and are not recorded). */
int k3moe_cache_trace_record(k3moe_cache *C, int32_t on);

/* The record so far: *host_n_keys / *host_n_batches receive its sizes; the
 * keys and batch lengths are copied out when the host arrays are non-null
 * and large enough (cap_keys, cap_batches), else K3MOE_EINVAL. */
int k3moe_cache_trace_get(const k3moe_cache *C, int64_t *host_keys, int64_t cap_keys,
                          int32_t *host_batch_len, int32_t cap_batches, int64_t *host_n_keys,
                          int32_t *host_n_batches);

/*
 * Replays a trace through a cache of `capacity` slots.  K3MOE_POLICY_LRU
 * makes exactly the live cache's decisions (hits first, then each miss takes
 * the lowest EMPTY slot, else the least recently used slot, lowest index on
 * ties, that is neither pinned nor used by the same batch; a key repeated in
 * a batch is a hit the second time); the npinned keys of host_pinned are
 * loaded first, into slots 0..npinned-1, and never evicted.
 * K3MOE_POLICY_BELADY evicts the resident key, not used by the same batch,
 * whose next use is farthest away (npinned must be 0).
 *  host_hit_out  optional uint8 per trace key: 1 hit, 0 miss
 *  host_hits_out receives the hit count
 * K3MOE_EBUSY if a batch finds no evictable slot, K3MOE_EINVAL on bad
 * arguments (a negative key, batch_len < 1, npinned > capacity).
 */
int k3moe_trace_replay(const int64_t *host_keys, const int32_t *host_batch_len, int32_t n_batches,
                       int32_t capacity, int32_t policy, const int64_t *host_pinned,
                       int32_t npinned, uint8_t *host_hit_out, int64_t *host_hits_out);

/* Cache sizing: the hit count at each of ncap capacities (replays run on
 * host threads); host_hits_out[c] is -1 where a batch does not fit. */
int k3moe_trace_sweep(const int64_t *host_keys, const int32_t *host_batch_len, int32_t n_batches,
                      const int32_t *host_capacities, int32_t ncap, int32_t policy,
                      int64_t *host_hits_out);

/* Sizing the pinned hot set: for each c < ncounts, the LRU replay of the
 * trace through `capacity` slots with hot_keys[0..pin_counts[c]) pinned (as
 * in k3moe_trace_replay), counting only the hits at trace positions >=
 * count_from (e.g. a hot set measured on the first part of a trace and judged
 * on the rest).  host_hits_out[c] is -1 where a batch does not fit.  Replays
 * run on host threads. */
int k3moe_trace_pin_sweep(const int64_t *host_keys, const int32_t *host_batch_len, int32_t n_batches,
                          int32_t capacity, const int64_t *host_hot_keys,
                          const int32_t *host_pin_counts, int32_t ncounts, int64_t count_from,
                          int64_t *host_hits_out);

/* Hot set: the n keys with the largest counts in hist[0..nkeys), in order of
 * decreasing count, ties to the lower key.  K3MOE_EINVAL if n > nkeys. */
int k3moe_hot_set(const uint32_t *host_hist, int64_t nkeys, int32_t n, int64_t *host_keys_out);

/* Pins the n most requested keys of the cache's own histogram (hottest
 * first; K3MOE_EBUSY from the first that finds no slot). */
int k3moe_cache_pin_hot(k3moe_cache *C, int32_t n, k3moe_stream compute);

/* Ends a pin: the key stays cached and becomes evictable again (no-op for a
 * key that is not pinned). */
int k3moe_cache_unpin(k3moe_cache *C, int64_t key);

/* Trace file: "K3TRACE1", int64 n_batches, int64 n_keys, int32
 * batch_len[n_batches], int64 keys[n_keys], little-endian.  load with null
 * arrays reports the sizes only; K3MOE_EINVAL for a file that is not such a
 * trace (or arrays too small), K3MOE_EIO if it cannot be opened or written. */
int k3moe_trace_save(const char *path, const int64_t *host_keys, const int32_t *host_batch_len,
                     int32_t n_batches);
int k3moe_trace_load(const char *path, int64_t *host_keys, int64_t cap_keys,
                     int32_t *host_batch_len, int32_t cap_batches, int64_t *host_n_keys,
                     int32_t *host_n_batches);

/* ------------------------------------------ shared (always-on) experts */

/*
 * A shared expert of the dense trunk: each MoE layer of the pages' model has
 * two that run on every token next to the routed ones ["Running Kimi K3
 * locally", "What are the four reductions, and why is the answer
 * unchanged?"], kept in bf16 like the rest of the trunk ["kimi-k3-in-c"
 * explainer, "Why the trunk stays at 16 bits"].  Row-major bf16 bit
 * patterns: gate, up [f][d], down [d][f]; each pointer 16-byte aligned.
 * A blob of k3moe_shared_expert_bytes(d, f) = 6 d f bytes holds gate, up
 * and down in that order (k3moe_shared_expert_view).
 */
typedef struct {
    const uint16_t *gate, *up, *down;
} k3moe_bf16_expert;

#define K3MOE_MAX_SHARED 4
int64_t k3moe_shared_expert_bytes(int32_t d, int32_t f);
int k3moe_shared_expert_view(k3moe_bf16_expert *host_out, const void *blob, int32_t d, int32_t f);
/* Workspace bytes of k3moe_shared_forward for n_shared experts of size f. */
size_t k3moe_shared_workspace(int32_t n_shared, int32_t f);
/*
 * out[t] (+)= sum_s W_down^s (silu(W_gate^s x_t) * (W_up^s x_t)) for the
 * n_shared (1..K3MOE_MAX_SHARED) experts: the shared experts' outputs are
 * added with weight 1 (a reading: the pages do not say how they combine;
 * an always-on expert has no router weight).  fp32 accumulation.
 *  x, out     device fp32 [T][d]; accumulate != 0 adds into out
 *  d, f       multiples of 256, d <= 8192 and n_shared * f <= 4096 (the
 *             lanes of a warp hold a whole down row of the n_shared experts)
 *  workspace  device, k3moe_shared_workspace(n_shared, f) bytes
 * Errors: K3MOE_EINVAL for null or misaligned pointers, bad sizes.
 */
int k3moe_shared_forward(float *out, const float *x, int32_t T, const k3moe_bf16_expert *host_experts,
                         int32_t n_shared, int32_t d, int32_t f, int32_t accumulate, void *workspace,
                         size_t workspace_bytes, k3moe_stream s);

/* ------------------------------------------------ dense trunk streaming */

/*
 * Per-layer weights that every token reads in the same order (the pages'
 * dense trunk: layer 0, 1, ..., M-1 on every token) kept as a pinned prefix
 * plus a ring of streaming slots [LOCAL, "the four reductions", reduction
 * three; ENG, "The interesting design decisions"]: a cyclic scan defeats
 * LRU (an LRU of C < M slots hits nothing), while a resident prefix of P
 * layers hits exactly P/M.
 *
 *  host_layers[M]       host pointers to each layer's bytes (pinned by the
 *                       caller for full speed), host_layer_bytes[M] sizes
 *                       (each > 0, a multiple of 16)
 *  pinned_bytes         HBM budget of the prefix: layers 0..P-1 are resident,
 *                       P the largest count whose sizes (rounded up to 256 B)
 *                       fit; they are copied once, stream-ordered
 *  ring_slots           R streaming slots of the largest streamed layer's
 *                       size; R >= 1 when P < M (R >= 2 lets the next layer
 *                       copy while the current one computes)
 *
 * The streamed layers P..M-1 are expected in cyclic order (after M-1 comes
 * P of the next token).  The n-th streamed request uses ring slot n mod R;
 * after each acquire and release the copies of the next layers are issued
 * into free slots (at most R - 1 ahead), each after the release of the
 * slot's previous layer.  A request out of that order is served too, with
 * its copy issued on demand.  A failed prefetch copy is not an error of the
 * call that issued it: the layer is copied again when it is requested, and
 * that request returns the copier's code if the copy fails again.
 */
typedef struct k3moe_trunk k3moe_trunk;

typedef struct {
    int64_t requests;       /* acquires                                       */
    int64_t resident;       /* acquires of prefix layers                      */
    int64_t prefetched;     /* streamed acquires whose copy was already issued */
    int64_t h2d_bytes;      /* bytes copied host -> HBM (prefix included)     */
    int32_t n_layers;
    int32_t pinned_layers;  /* P */
    int32_t ring_slots;     /* R */
    int32_t reserved;
} k3moe_trunk_stats;

int k3moe_trunk_create(k3moe_trunk **host_out, const void *const *host_layers,
                       const size_t *host_layer_bytes, int32_t n_layers, size_t pinned_bytes,
                       int32_t ring_slots);
/* The same over a copier (k3moe_copier below the cache): copier slots
 * 0..P-1 are the prefix layers, P..P+R-1 the ring.  No CUDA call. */
int k3moe_trunk_create_with_copier(k3moe_trunk **host_out, const void *const *host_layers,
                                   const size_t *host_layer_bytes, int32_t n_layers,
                                   size_t pinned_bytes, int32_t ring_slots,
                                   const k3moe_copier *host_copier);
int k3moe_trunk_destroy(k3moe_trunk *T);

/* Device pointer of `layer`'s bytes, usable on `compute` (which is made to
 * wait for its copy).  host_resident_out (optional) receives 1 for a prefix
 * layer.  The layer stays valid until k3moe_trunk_release.  K3MOE_EBUSY if
 * its ring slot still holds a layer that has not been released. */
int k3moe_trunk_acquire(k3moe_trunk *T, int32_t layer, void **host_dev_out,
                        uint8_t *host_resident_out, k3moe_stream compute);
/* Ends the use of an acquired layer: records on `compute` the point after
 * which its ring slot may be overwritten (no-op for a prefix layer). */
int k3moe_trunk_release(k3moe_trunk *T, int32_t layer, k3moe_stream compute);
int k3moe_trunk_get_stats(const k3moe_trunk *T, k3moe_trunk_stats *host_out);

/* --------------------------------------------------- streamed decode loop */

/*
 * Batch-1 decode of T tokens through n_layers MoE layers whose experts live
 * in host memory behind an expert cache (the pages' streaming design [EXPL,
 * "The cache the project exists for"; HOW, "The LRU cache"], with the host
 * pool in pinned RAM instead of NVMe).  For every token t and layer l:
 *   u   = x / sqrt(mean(x^2) + eps)                 (RMSNorm, unit gain)
 *   ids, w = top-k routing of u by layer l's router (+ selection bias)
 *   the k ids go to the host (one small D2H copy; the stream is synchronised)
 *   slots = k3moe_cache_acquire_split(keys l * n_experts + ids)
 *   x  += sum over hits of w_j * expert_{ids_j}(u)   (while the misses copy)
 *   for each miss j, in copy order:
 *       k3moe_cache_wait_copy(slot j);  x += w_j * expert_{ids_j}(u)
 *   k3moe_cache_release
 *   with desc.trunk: x += sum_s shared_expert_s(u), the n_shared bf16 shared
 *   experts of layer l read from trunk layer l (k3moe_trunk_acquire /
 *   _release; n_shared consecutive blobs of k3moe_shared_expert_bytes(d, f))
 *  desc.host_layers  host array of n_layers layers (router-only layers are
 *                    fine: created with host_experts = NULL); all with the
 *                    same n_experts, top_k, d, f; top_k <= 16
 *  desc.cache        keys layer * n_experts + expert, blobs of
 *                    k3moe_expert_bytes(d, f)
 *  X  fp32 [T x d] input hidden states, out fp32 [T x d] after the last layer
 *  host_ids_out  optional int32 [T][n_layers][top_k] (ascending ids)
 *  host_hit_out  optional uint8 [T][n_layers][top_k] cache hit flags
 * Returns the first failing status (the cache's K3MOE_EBUSY included).
 */
typedef struct {
    int32_t n_layers;
    k3moe_layer *const *host_layers;
    k3moe_cache *cache;
    float eps;
    k3moe_trunk *trunk;  /* optional: layer l's trunk bytes hold its shared experts */
    int32_t n_shared;    /* shared experts per layer (0 without a trunk)           */
} k3moe_stream_desc;

int k3moe_stream_decode(const k3moe_stream_desc *host_desc, const float *X, int32_t T, float *out,
                        int32_t *host_ids_out, uint8_t *host_hit_out, k3moe_stream s);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */
