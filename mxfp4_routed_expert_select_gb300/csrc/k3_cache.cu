// k3_cache.cu -- HBM-resident LRU expert cache fed from pinned host memory.
//
// What the pages describe for the CPU engine's expert cache ("kimi-k3-in-c"
// explainer, "The cache the project exists for" and "The bug the code
// confesses to"; "How kimi-k3-in-c Runs...", "The LRU cache"), rebuilt for
// one GPU: the arena is one cudaMalloc of `slots` expert blobs in HBM; a miss
// is one cudaMemcpyAsync of the expert's blob on a side stream; the caller's
// compute stream waits on per-slot events, so the host never blocks.  The
// copies of one batch go to one side stream, in the batch's order, so that
// they land one after the other and a caller can compute on each as soon as
// it is in (a measured host link gives the same ~200 GB/s to one stream as
// to several); successive batches take the side streams in turn.
//
// Slot states: a key (>= 0), EMPTY, or INFLIGHT.  INFLIGHT marks a slot that
// a batch has reserved for a copy and not yet published.  Victim selection
// skips INFLIGHT slots, so two misses of one batch can never be given the
// same slot -- the failure the explainer page reports for the CPU engine,
// where an "empty" fast path handed one slot to several parallel reads.
//
// Replacement: a batch's hits are marked first (most recently used, in use);
// each miss then takes the lowest-index EMPTY slot, else the least recently
// used slot (lowest index on ties) that is neither pinned nor in use.  Slots
// stay "in use" from acquire until k3moe_cache_release, which records on the
// compute stream the point after which they may be overwritten.
#include <cuda_runtime.h>

#include <cstring>
#include <exception>
#include <new>
#include <utility>
#include <vector>

#include "k3moe.h"

namespace {

constexpr int64_t kEmpty = -1;
constexpr int64_t kInflight = -2;

// Default copier: device arena, side streams, per-slot copy/release events.
constexpr int kSideStreams = 4;
struct CudaCopier {
    cudaStream_t side[kSideStreams] = {};
    unsigned next = 0;               // side stream of the next batch
    unsigned cur = 0;                // side stream of this batch
    cudaStream_t compute = nullptr;  // set per call
    std::vector<cudaEvent_t> copied, released;
    std::vector<char> has_release;
};

int cuda_alloc(void *ctx, size_t bytes, void **out)
{
    (void)ctx;
    if (cudaMalloc(out, bytes) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ENOMEM;
    }
    return K3MOE_OK;
}
int cuda_free(void *ctx, void *p)
{
    (void)ctx;
    return cudaFree(p) == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}
int cuda_copy(void *ctx, int32_t slot, void *dst, const void *src, size_t bytes)
{
    CudaCopier *c = (CudaCopier *)ctx;
    cudaStream_t side = c->side[c->cur];
    if (c->has_release[slot] && cudaStreamWaitEvent(side, c->released[slot], 0) != cudaSuccess)
        return K3MOE_ECUDA;
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, side) != cudaSuccess) return K3MOE_ECUDA;
    if (cudaEventRecord(c->copied[slot], side) != cudaSuccess) return K3MOE_ECUDA;
    return K3MOE_OK;
}
int cuda_wait(void *ctx, int32_t slot)
{
    CudaCopier *c = (CudaCopier *)ctx;
    return cudaStreamWaitEvent(c->compute, c->copied[slot], 0) == cudaSuccess ? K3MOE_OK
                                                                               : K3MOE_ECUDA;
}
int cuda_release(void *ctx, int32_t slot)
{
    CudaCopier *c = (CudaCopier *)ctx;
    if (cudaEventRecord(c->released[slot], c->compute) != cudaSuccess) return K3MOE_ECUDA;
    c->has_release[slot] = 1;
    return K3MOE_OK;
}

}  // namespace

struct k3moe_cache {
    size_t expert_bytes = 0;
    int32_t n_layers = 0, n_experts = 0;
    int64_t nkeys = 0;
    std::vector<const void *> host;
    int32_t slots = 0;
    uint8_t *arena = nullptr;
    std::vector<int64_t> key;       // per slot: key, kEmpty or kInflight
    std::vector<int64_t> last;      // per slot: recency stamp
    std::vector<uint8_t> pin;       // per slot
    std::vector<int32_t> in_use;    // per slot: acquired and not released
    std::vector<int32_t> where;     // per key: slot or -1
    std::vector<uint32_t> hist;     // per key: requests
    k3moe_cache_stats st;
    int64_t now = 0;
    k3moe_copier cp;
    CudaCopier *cuda = nullptr;     // when the default copier is used
    std::vector<int32_t> used;      // slots handed out since the last release
    std::vector<std::pair<int32_t, int64_t>> pending;  // (slot, key) copied, not waited for
    bool tracing = false;           // record the keys of every placed batch
    std::vector<int64_t> trace_keys;
    std::vector<int32_t> trace_len;
};

static void cache_free(k3moe_cache *C)
{
    if (!C) return;
    if (C->arena) C->cp.free_arena(C->cp.ctx, C->arena);
    if (C->cuda) {
        for (auto e : C->cuda->copied)
            if (e) cudaEventDestroy(e);
        for (auto e : C->cuda->released)
            if (e) cudaEventDestroy(e);
        for (cudaStream_t st : C->cuda->side)
            if (st) cudaStreamDestroy(st);
        delete C->cuda;
    }
    delete C;
}

static int cache_init(k3moe_cache **out, size_t capacity_bytes, size_t expert_bytes,
                      const void *const *host_blobs, int32_t n_layers, int32_t n_experts,
                      const k3moe_copier *cp, bool use_cuda)
{
    if (!out) return K3MOE_EINVAL;
    *out = nullptr;
    if (expert_bytes == 0 || expert_bytes % 16 || !host_blobs || n_layers <= 0 || n_experts <= 0)
        return K3MOE_EINVAL;
    const size_t slots = capacity_bytes / expert_bytes;
    if (slots < 1 || slots > (1u << 30)) return K3MOE_EINVAL;
    const int64_t nkeys = (int64_t)n_layers * n_experts;
    for (int64_t q = 0; q < nkeys; q++)
        if (!host_blobs[q]) return K3MOE_EINVAL;
    k3moe_cache *C = new (std::nothrow) k3moe_cache;
    if (!C) return K3MOE_ENOMEM;
    C->expert_bytes = expert_bytes;
    C->n_layers = n_layers;
    C->n_experts = n_experts;
    C->nkeys = nkeys;
    C->slots = (int32_t)slots;
    try {
        C->host.assign(host_blobs, host_blobs + nkeys);
        C->key.assign(slots, kEmpty);
        C->last.assign(slots, -1);
        C->pin.assign(slots, 0);
        C->in_use.assign(slots, 0);
        C->where.assign(nkeys, -1);
        C->hist.assign(nkeys, 0);
        C->used.reserve(slots);     // at most one entry per slot
        C->pending.reserve(slots);  // an INFLIGHT slot is never a victim
    } catch (const std::exception &) {
        delete C;
        return K3MOE_ENOMEM;
    }
    memset(&C->st, 0, sizeof(C->st));
    C->st.slots = C->slots;
    if (use_cuda) {
        C->cuda = new (std::nothrow) CudaCopier;
        if (!C->cuda) {
            delete C;
            return K3MOE_ENOMEM;
        }
        C->cp = {C->cuda, cuda_alloc, cuda_free, cuda_copy, cuda_wait, cuda_release};
        for (cudaStream_t &st : C->cuda->side)
            if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
                cudaGetLastError();
                cache_free(C);
                return K3MOE_ECUDA;
            }
        try {
            C->cuda->copied.assign(slots, nullptr);
            C->cuda->released.assign(slots, nullptr);
            C->cuda->has_release.assign(slots, 0);
        } catch (const std::exception &) {
            cache_free(C);
            return K3MOE_ENOMEM;
        }
        for (size_t s = 0; s < slots; s++) {
            if (cudaEventCreateWithFlags(&C->cuda->copied[s], cudaEventDisableTiming) !=
                    cudaSuccess ||
                cudaEventCreateWithFlags(&C->cuda->released[s], cudaEventDisableTiming) !=
                    cudaSuccess) {
                cudaGetLastError();
                cache_free(C);
                return K3MOE_ECUDA;
            }
        }
    } else {
        C->cp = *cp;
    }
    void *arena = nullptr;
    int rc = C->cp.alloc_arena(C->cp.ctx, slots * expert_bytes, &arena);
    if (rc != K3MOE_OK || !arena) {
        cache_free(C);
        return rc != K3MOE_OK ? rc : K3MOE_ENOMEM;
    }
    C->arena = (uint8_t *)arena;
    *out = C;
    return K3MOE_OK;
}

// Victim for one miss: lowest-index EMPTY slot, else the least recently used
// slot that is not pinned, not in use and not INFLIGHT.  `taken` marks slots
// already planned for this batch.
static int32_t pick_victim(const k3moe_cache *C, const std::vector<char> &taken)
{
    for (int32_t s = 0; s < C->slots; s++)
        if (!taken[s] && C->key[s] == kEmpty) return s;
    int32_t v = -1;
    for (int32_t s = 0; s < C->slots; s++) {
        if (taken[s] || C->pin[s] || C->in_use[s] || C->key[s] == kInflight) continue;
        if (v < 0 || C->last[s] < C->last[v]) v = s;
    }
    return v;
}

extern "C" {

int k3moe_cache_create(k3moe_cache **out, size_t capacity_bytes, size_t expert_bytes,
                       const void *const *host_blobs, int32_t n_layers, int32_t n_experts)
{
    return cache_init(out, capacity_bytes, expert_bytes, host_blobs, n_layers, n_experts, nullptr,
                      true);
}

int k3moe_cache_create_with_copier(k3moe_cache **out, size_t capacity_bytes,
                                   size_t expert_bytes, const void *const *host_blobs,
                                   int32_t n_layers, int32_t n_experts, const k3moe_copier *cp)
{
    if (!cp || !cp->alloc_arena || !cp->free_arena || !cp->copy || !cp->wait || !cp->release)
        return K3MOE_EINVAL;
    return cache_init(out, capacity_bytes, expert_bytes, host_blobs, n_layers, n_experts, cp,
                      false);
}

int k3moe_cache_destroy(k3moe_cache *C)
{
    if (!C) return K3MOE_EINVAL;
    if (C->cuda)
        for (cudaStream_t st : C->cuda->side)
            if (st) cudaStreamSynchronize(st);
    cache_free(C);
    return K3MOE_OK;
}

// Makes `compute` wait for the copy into slot s (an INFLIGHT slot) and
// publishes its key.
static int wait_one(k3moe_cache *C, int32_t s, int64_t key)
{
    if (C->key[s] != kInflight) return K3MOE_OK;
    const int r = C->cp.wait(C->cp.ctx, s);
    if (r != K3MOE_OK) {
        C->key[s] = kEmpty;
        return r;
    }
    C->key[s] = key;
    C->where[key] = s;
    return K3MOE_OK;
}

// Makes `compute` wait for every copy issued and not yet waited for, and
// publishes those slots' keys (INFLIGHT -> key).
static int wait_pending(k3moe_cache *C, k3moe_stream compute)
{
    if (C->cuda) C->cuda->compute = reinterpret_cast<cudaStream_t>(compute);
    int rc = K3MOE_OK;
    for (const auto &pk : C->pending) {
        const int r = wait_one(C, pk.first, pk.second);
        if (r != K3MOE_OK && rc == K3MOE_OK) rc = r;
    }
    C->pending.clear();
    return rc;
}

static int acquire(k3moe_cache *C, const int64_t *keys, int32_t n, void **blobs_out,
                   uint8_t *hit_out, k3moe_stream compute, bool wait)
{
    if (!C || !keys || !blobs_out || n <= 0) return K3MOE_EINVAL;
    for (int32_t i = 0; i < n; i++)
        if (keys[i] < 0 || keys[i] >= C->nkeys) return K3MOE_EINVAL;
    // copies of an earlier split acquire are published first, so that their
    // keys are found as hits and not copied a second time
    int rc = wait_pending(C, compute);

    // plan: hits, then one distinct victim per distinct missing key
    std::vector<char> taken(C->slots, 0);
    std::vector<int32_t> slot_of(n, -1);
    std::vector<char> is_hit(n, 0);
    for (int32_t i = 0; i < n; i++) {
        const int32_t s = C->where[keys[i]];
        if (s >= 0) {
            slot_of[i] = s;
            is_hit[i] = 1;
            taken[s] = 1;
        }
    }
    std::vector<int32_t> victims;
    for (int32_t i = 0; i < n; i++) {
        if (slot_of[i] >= 0) continue;
        int32_t dup = -1;
        for (int32_t q = 0; q < i; q++)
            if (keys[q] == keys[i] && slot_of[q] >= 0) { dup = slot_of[q]; break; }
        if (dup >= 0) {
            slot_of[i] = dup;
            is_hit[i] = 1;  // a repeated key is a hit the second time
            continue;
        }
        const int32_t v = pick_victim(C, taken);
        if (v < 0) return K3MOE_EBUSY;  // nothing committed yet
        taken[v] = 1;
        slot_of[i] = v;
        victims.push_back(i);
    }

    // the record of the trace grows before anything is committed, so that a
    // failed allocation leaves the cache as it was
    if (C->tracing) {
        const size_t nk = C->trace_keys.size();
        try {
            C->trace_keys.insert(C->trace_keys.end(), keys, keys + n);
            C->trace_len.push_back(n);
        } catch (const std::exception &) {
            C->trace_keys.resize(nk);
            return K3MOE_ENOMEM;
        }
    }
    // commit (no allocation below: used and pending hold at most one entry
    // per slot and were reserved at create): recency and use marks for every
    // slot of the batch
    for (int32_t i = 0; i < n; i++) {
        C->hist[keys[i]]++;
        const int32_t s = slot_of[i];
        C->last[s] = C->now;
        if (!C->in_use[s]) C->used.push_back(s);
        C->in_use[s] = 1;
    }
    for (int32_t i : victims) {
        const int32_t s = slot_of[i];
        if (C->key[s] >= 0) {
            C->where[C->key[s]] = -1;
            C->st.evictions++;
        }
        C->key[s] = kInflight;
    }
    if (C->cuda && !victims.empty()) C->cuda->cur = C->cuda->next++ % kSideStreams;
    for (int32_t i : victims) {
        const int32_t s = slot_of[i];
        int r = C->cp.copy(C->cp.ctx, s, C->arena + (size_t)s * C->expert_bytes, C->host[keys[i]],
                           C->expert_bytes);
        if (r != K3MOE_OK) {
            C->key[s] = kEmpty;
            if (rc == K3MOE_OK) rc = r;
            continue;
        }
        C->st.h2d_bytes += (int64_t)C->expert_bytes;
        C->pending.emplace_back(s, keys[i]);
    }
    if (wait) {
        const int r = wait_pending(C, compute);
        if (rc == K3MOE_OK) rc = r;
    }
    for (int32_t i = 0; i < n; i++) {
        blobs_out[i] = C->arena + (size_t)slot_of[i] * C->expert_bytes;
        if (hit_out) hit_out[i] = is_hit[i];
    }
    int64_t nh = 0;
    for (int32_t i = 0; i < n; i++) nh += is_hit[i];
    C->st.lookups += n;
    C->st.hits += nh;
    C->st.misses += n - nh;
    C->st.hbm_bytes += (int64_t)n * (int64_t)C->expert_bytes;
    C->now++;
    return rc;
}

// The plan's scratch vectors are allocated before anything is committed: a
// failed allocation changes nothing.
static int acquire_guarded(k3moe_cache *C, const int64_t *keys, int32_t n, void **blobs_out,
                           uint8_t *hit_out, k3moe_stream compute, bool wait)
{
    try {
        return acquire(C, keys, n, blobs_out, hit_out, compute, wait);
    } catch (const std::exception &) {
        return K3MOE_ENOMEM;
    }
}

int k3moe_cache_acquire(k3moe_cache *C, const int64_t *keys, int32_t n, void **blobs_out,
                        uint8_t *hit_out, k3moe_stream compute)
{
    return acquire_guarded(C, keys, n, blobs_out, hit_out, compute, true);
}

int k3moe_cache_acquire_split(k3moe_cache *C, const int64_t *keys, int32_t n, void **blobs_out,
                              uint8_t *hit_out, k3moe_stream compute)
{
    return acquire_guarded(C, keys, n, blobs_out, hit_out, compute, false);
}

int k3moe_cache_wait_copies(k3moe_cache *C, k3moe_stream compute)
{
    if (!C) return K3MOE_EINVAL;
    return wait_pending(C, compute);
}

int k3moe_cache_wait_copy(k3moe_cache *C, const void *blob, k3moe_stream compute)
{
    if (!C || !blob) return K3MOE_EINVAL;
    const uint8_t *b = (const uint8_t *)blob;
    if (b < C->arena) return K3MOE_EINVAL;
    const size_t off = (size_t)(b - C->arena);
    if (off % C->expert_bytes || off / C->expert_bytes >= (size_t)C->slots) return K3MOE_EINVAL;
    const int32_t s = (int32_t)(off / C->expert_bytes);
    for (size_t q = 0; q < C->pending.size(); q++) {
        if (C->pending[q].first != s) continue;
        if (C->cuda) C->cuda->compute = reinterpret_cast<cudaStream_t>(compute);
        const int r = wait_one(C, s, C->pending[q].second);
        C->pending.erase(C->pending.begin() + (long)q);
        return r;
    }
    return K3MOE_OK;  // a hit, or a copy already waited for
}

int k3moe_cache_release(k3moe_cache *C, k3moe_stream compute)
{
    if (!C) return K3MOE_EINVAL;
    // a slot whose copy `compute` has not waited for must not be marked free
    // on `compute`: the next copy into it could overtake the running one
    int rc = wait_pending(C, compute);
    for (int32_t s : C->used) {
        int r = C->cp.release(C->cp.ctx, s);
        if (r != K3MOE_OK && rc == K3MOE_OK) rc = r;
        C->in_use[s] = 0;
    }
    C->used.clear();
    return rc;
}

int k3moe_cache_pin(k3moe_cache *C, int64_t key, k3moe_stream compute)
{
    if (!C || key < 0 || key >= C->nkeys) return K3MOE_EINVAL;
    void *blob = nullptr;
    // pinning is not a request: keep the request counters as they were
    const k3moe_cache_stats before = C->st;
    const uint32_t h = C->hist[key];
    const bool tracing = C->tracing;
    C->tracing = false;
    int rc = k3moe_cache_acquire(C, &key, 1, &blob, nullptr, compute);
    C->tracing = tracing;
    C->st.lookups = before.lookups;
    C->st.hits = before.hits;
    C->st.misses = before.misses;
    C->st.hbm_bytes = before.hbm_bytes;
    C->hist[key] = h;
    if (rc != K3MOE_OK) return rc;
    const int32_t s = C->where[key];
    if (s >= 0 && !C->pin[s]) {
        C->pin[s] = 1;
        C->st.pinned++;
    }
    return k3moe_cache_release(C, compute);
}

int k3moe_cache_pin_hot(k3moe_cache *C, int32_t n, k3moe_stream compute)
{
    if (!C || n < 0 || n > C->nkeys) return K3MOE_EINVAL;
    std::vector<int64_t> hot((size_t)n);
    int rc = k3moe_hot_set(C->hist.data(), C->nkeys, n, hot.data());
    for (int32_t i = 0; i < n && rc == K3MOE_OK; i++) rc = k3moe_cache_pin(C, hot[(size_t)i], compute);
    return rc;
}

int k3moe_cache_unpin(k3moe_cache *C, int64_t key)
{
    if (!C || key < 0 || key >= C->nkeys) return K3MOE_EINVAL;
    const int32_t s = C->where[key];
    if (s >= 0 && C->pin[s]) {
        C->pin[s] = 0;
        C->st.pinned--;
    }
    return K3MOE_OK;
}

int k3moe_cache_trace_record(k3moe_cache *C, int32_t on)
{
    if (!C) return K3MOE_EINVAL;
    if (on) {
        C->trace_keys.clear();
        C->trace_len.clear();
    }
    C->tracing = on != 0;
    return K3MOE_OK;
}

int k3moe_cache_trace_get(const k3moe_cache *C, int64_t *keys, int64_t cap_keys, int32_t *batch_len,
                          int32_t cap_batches, int64_t *n_keys, int32_t *n_batches)
{
    if (!C || !n_keys || !n_batches) return K3MOE_EINVAL;
    const int64_t nk = (int64_t)C->trace_keys.size();
    const int32_t nb = (int32_t)C->trace_len.size();
    *n_keys = nk;
    *n_batches = nb;
    if (keys) {
        if (cap_keys < nk) return K3MOE_EINVAL;
        if (nk) memcpy(keys, C->trace_keys.data(), sizeof(int64_t) * (size_t)nk);
    }
    if (batch_len) {
        if (cap_batches < nb) return K3MOE_EINVAL;
        if (nb) memcpy(batch_len, C->trace_len.data(), sizeof(int32_t) * (size_t)nb);
    }
    return K3MOE_OK;
}

int k3moe_cache_get_stats(k3moe_cache *C, k3moe_cache_stats *out)
{
    if (!C || !out) return K3MOE_EINVAL;
    *out = C->st;
    int32_t inflight = 0;
    for (int32_t s = 0; s < C->slots; s++) inflight += (C->key[s] == kInflight);
    out->inflight = inflight;
    return K3MOE_OK;
}

const uint32_t *k3moe_cache_histogram(const k3moe_cache *C) { return C ? C->hist.data() : nullptr; }

int32_t k3moe_cache_slot_of(const k3moe_cache *C, int64_t key)
{
    if (!C || key < 0 || key >= C->nkeys) return -1;
    return C->where[key];
}

}  // extern "C"
