// k3_trunk.cpp -- per-layer weights read in the same order on every token,
// kept as a resident prefix in HBM plus a ring of streaming slots.
//
// The pages stream their 108.81 GB dense trunk as a pinned prefix plus one
// ring slot ("Running Kimi K3 locally", the four reductions, reduction
// three): layers are walked 0..M-1 on every token, a cyclic scan, for which
// LRU is the worst policy (C < M slots hit nothing) and a resident prefix of
// P layers hits exactly P/M ("kimi-k3-in-c: A 176 KB Engine...", "The
// interesting design decisions").  On one GPU the prefix lives in HBM, the
// streamed layers come from host memory by cudaMemcpyAsync on a side stream,
// and with R >= 2 ring slots the copy of the next layer overlaps the compute
// on the current one.
//
// Streamed requests are numbered in the cyclic order (sequence q is layer
// P + q mod (M - P)); sequence q uses ring slot q mod R.  After every acquire
// and release the copies of the next sequences are issued, at most R - 1
// ahead of the next expected one, each into a slot whose previous layer has
// been released (the copy waits for that release on the device).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <exception>
#include <new>
#include <vector>

#include "k3moe.h"

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Default copier: one side stream (copies land in the order issued), a copy
// and a release event per slot.
struct TrunkCuda {
    cudaStream_t side = nullptr;
    cudaStream_t compute = nullptr;  // set per call
    std::vector<cudaEvent_t> copied, released;
    std::vector<char> has_release;
};

int tc_alloc(void *, size_t bytes, void **out)
{
    if (cudaMalloc(out, bytes) != cudaSuccess) {
        cudaGetLastError();
        return K3MOE_ENOMEM;
    }
    return K3MOE_OK;
}
int tc_free(void *, void *p) { return cudaFree(p) == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA; }
int tc_copy(void *ctx, int32_t slot, void *dst, const void *src, size_t bytes)
{
    TrunkCuda *c = (TrunkCuda *)ctx;
    if (c->has_release[slot] && cudaStreamWaitEvent(c->side, c->released[slot], 0) != cudaSuccess)
        return K3MOE_ECUDA;
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, c->side) != cudaSuccess) return K3MOE_ECUDA;
    return cudaEventRecord(c->copied[slot], c->side) == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}
int tc_wait(void *ctx, int32_t slot)
{
    TrunkCuda *c = (TrunkCuda *)ctx;
    return cudaStreamWaitEvent(c->compute, c->copied[slot], 0) == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}
int tc_release(void *ctx, int32_t slot)
{
    TrunkCuda *c = (TrunkCuda *)ctx;
    if (cudaEventRecord(c->released[slot], c->compute) != cudaSuccess) return K3MOE_ECUDA;
    c->has_release[slot] = 1;
    return K3MOE_OK;
}

}  // namespace

struct k3moe_trunk {
    int32_t M = 0, P = 0, R = 0;
    std::vector<const void *> host;
    std::vector<size_t> bytes;
    uint8_t *arena = nullptr;
    std::vector<size_t> off;            // per prefix layer: offset in the arena
    size_t ring_off = 0, ring_bytes = 0;
    std::vector<char> prefix_pending;   // prefix copy not yet waited for
    std::vector<int64_t> slot_seq;      // per ring slot: sequence held, or -1
    std::vector<char> slot_pending;     // copy issued, not waited for
    std::vector<char> slot_in_use;      // acquired, not released
    int64_t next_seq = 0;               // the next expected streamed sequence
    int64_t issued = 0;                 // copies issued for sequences < issued
    k3moe_trunk_stats st;
    k3moe_copier cp;
    TrunkCuda *cuda = nullptr;
};

static int32_t layer_of(const k3moe_trunk *T, int64_t q) { return T->P + (int32_t)(q % (T->M - T->P)); }
static uint8_t *slot_ptr(const k3moe_trunk *T, int32_t s) { return T->arena + T->ring_off + (size_t)s * T->ring_bytes; }

static int issue(k3moe_trunk *T, int64_t q)
{
    const int32_t s = (int32_t)(q % T->R), l = layer_of(T, q);
    const int r = T->cp.copy(T->cp.ctx, T->P + s, slot_ptr(T, s), T->host[(size_t)l], T->bytes[(size_t)l]);
    if (r != K3MOE_OK) {
        T->slot_seq[(size_t)s] = -1;
        T->slot_pending[(size_t)s] = 0;
        return r;
    }
    T->slot_seq[(size_t)s] = q;
    T->slot_pending[(size_t)s] = 1;
    T->st.h2d_bytes += (int64_t)T->bytes[(size_t)l];
    return K3MOE_OK;
}

// Copies of the sequences after the next expected one, into released slots.
// A failed copy stops the window there; its layer is copied again when it is
// requested, and that request reports the copier's code if it fails again.
static int prefetch(k3moe_trunk *T)
{
    if (T->issued < T->next_seq) T->issued = T->next_seq;
    while (T->issued < T->next_seq + T->R - 1) {
        const int32_t s = (int32_t)(T->issued % T->R);
        if (T->slot_in_use[(size_t)s]) break;
        const int r = issue(T, T->issued);
        if (r != K3MOE_OK) return r;
        T->issued++;
    }
    return K3MOE_OK;
}

static void trunk_free(k3moe_trunk *T)
{
    if (!T) return;
    if (T->cuda && T->cuda->side) cudaStreamSynchronize(T->cuda->side);
    if (T->arena) T->cp.free_arena(T->cp.ctx, T->arena);
    if (T->cuda) {
        for (auto e : T->cuda->copied)
            if (e) cudaEventDestroy(e);
        for (auto e : T->cuda->released)
            if (e) cudaEventDestroy(e);
        if (T->cuda->side) cudaStreamDestroy(T->cuda->side);
        delete T->cuda;
    }
    delete T;
}

static int trunk_init(k3moe_trunk **out, const void *const *host, const size_t *bytes, int32_t M,
                      size_t pinned_bytes, int32_t R, const k3moe_copier *cp)
{
    if (!out) return K3MOE_EINVAL;
    *out = nullptr;
    if (!host || !bytes || M < 1 || R < 0) return K3MOE_EINVAL;
    for (int32_t l = 0; l < M; l++)
        if (!host[l] || bytes[l] == 0 || bytes[l] % 16) return K3MOE_EINVAL;
    int32_t P = 0;
    size_t used = 0;
    while (P < M && used + round_up(bytes[P]) <= pinned_bytes) used += round_up(bytes[P++]);
    if (P < M && R < 1) return K3MOE_EINVAL;
    if (P == M) R = 0;
    size_t ring_bytes = 0;
    for (int32_t l = P; l < M; l++) ring_bytes = std::max(ring_bytes, round_up(bytes[l]));

    k3moe_trunk *T = new (std::nothrow) k3moe_trunk;
    if (!T) return K3MOE_ENOMEM;
    T->M = M;
    T->P = P;
    T->R = R;
    T->ring_off = used;
    T->ring_bytes = ring_bytes;
    try {
        T->host.assign(host, host + M);
        T->bytes.assign(bytes, bytes + M);
        T->off.reserve((size_t)P);
        T->prefix_pending.assign((size_t)P, 0);
        T->slot_seq.assign((size_t)R, -1);
        T->slot_pending.assign((size_t)R, 0);
        T->slot_in_use.assign((size_t)R, 0);
    } catch (const std::exception &) {
        delete T;
        return K3MOE_ENOMEM;
    }
    memset(&T->st, 0, sizeof(T->st));
    T->st.n_layers = M;
    T->st.pinned_layers = P;
    T->st.ring_slots = R;
    if (cp) {
        T->cp = *cp;
    } else {
        T->cuda = new (std::nothrow) TrunkCuda;
        if (!T->cuda) {
            delete T;
            return K3MOE_ENOMEM;
        }
        T->cp = {T->cuda, tc_alloc, tc_free, tc_copy, tc_wait, tc_release};
        const size_t ns = (size_t)P + (size_t)R;
        try {
            T->cuda->copied.assign(ns, nullptr);
            T->cuda->released.assign(ns, nullptr);
            T->cuda->has_release.assign(ns, 0);
        } catch (const std::exception &) {
            trunk_free(T);
            return K3MOE_ENOMEM;
        }
        bool ok = cudaStreamCreateWithFlags(&T->cuda->side, cudaStreamNonBlocking) == cudaSuccess;
        for (size_t s = 0; ok && s < ns; s++)
            ok = cudaEventCreateWithFlags(&T->cuda->copied[s], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&T->cuda->released[s], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            trunk_free(T);
            return K3MOE_ECUDA;
        }
    }
    void *arena = nullptr;
    int rc = T->cp.alloc_arena(T->cp.ctx, used + (size_t)R * ring_bytes, &arena);
    if (rc != K3MOE_OK || !arena) {
        trunk_free(T);
        return rc != K3MOE_OK ? rc : K3MOE_ENOMEM;
    }
    T->arena = (uint8_t *)arena;
    // the prefix, copied once; each layer's first acquire waits for its copy
    size_t o = 0;
    for (int32_t l = 0; l < P && rc == K3MOE_OK; l++) {
        T->off.push_back(o);
        rc = T->cp.copy(T->cp.ctx, l, T->arena + o, host[l], bytes[l]);
        T->prefix_pending[(size_t)l] = 1;
        T->st.h2d_bytes += (int64_t)bytes[l];
        o += round_up(bytes[l]);
    }
    if (rc == K3MOE_OK && R > 0) prefetch(T);
    if (rc != K3MOE_OK) {
        trunk_free(T);
        return rc;
    }
    *out = T;
    return K3MOE_OK;
}

extern "C" {

int k3moe_trunk_create(k3moe_trunk **out, const void *const *host_layers, const size_t *layer_bytes,
                       int32_t n_layers, size_t pinned_bytes, int32_t ring_slots)
{
    return trunk_init(out, host_layers, layer_bytes, n_layers, pinned_bytes, ring_slots, nullptr);
}

int k3moe_trunk_create_with_copier(k3moe_trunk **out, const void *const *host_layers,
                                   const size_t *layer_bytes, int32_t n_layers, size_t pinned_bytes,
                                   int32_t ring_slots, const k3moe_copier *cp)
{
    if (!cp || !cp->alloc_arena || !cp->free_arena || !cp->copy || !cp->wait || !cp->release)
        return K3MOE_EINVAL;
    return trunk_init(out, host_layers, layer_bytes, n_layers, pinned_bytes, ring_slots, cp);
}

int k3moe_trunk_destroy(k3moe_trunk *T)
{
    if (!T) return K3MOE_EINVAL;
    trunk_free(T);
    return K3MOE_OK;
}

int k3moe_trunk_acquire(k3moe_trunk *T, int32_t layer, void **dev_out, uint8_t *resident_out,
                        k3moe_stream compute)
{
    if (!T || !dev_out || layer < 0 || layer >= T->M) return K3MOE_EINVAL;
    if (T->cuda) T->cuda->compute = reinterpret_cast<cudaStream_t>(compute);
    if (layer < T->P) {
        if (T->prefix_pending[(size_t)layer]) {
            const int r = T->cp.wait(T->cp.ctx, layer);
            if (r != K3MOE_OK) return r;
            T->prefix_pending[(size_t)layer] = 0;
        }
        T->st.requests++;
        T->st.resident++;
        *dev_out = T->arena + T->off[(size_t)layer];
        if (resident_out) *resident_out = 1;
        return K3MOE_OK;
    }
    // the first sequence at or after the expected one that holds this layer
    const int64_t S = T->M - T->P;
    const int64_t q = T->next_seq + ((layer - layer_of(T, T->next_seq)) % S + S) % S;
    const int32_t s = (int32_t)(q % T->R);
    const bool have = T->slot_seq[(size_t)s] == q;
    if (!have && T->slot_in_use[(size_t)s]) return K3MOE_EBUSY;  // nothing changed
    if (have) {
        T->st.prefetched++;
    } else {
        const int r = issue(T, q);
        if (r != K3MOE_OK) return r;
    }
    if (T->slot_pending[(size_t)s]) {
        const int r = T->cp.wait(T->cp.ctx, T->P + s);
        if (r != K3MOE_OK) {
            T->slot_seq[(size_t)s] = -1;
            T->slot_pending[(size_t)s] = 0;
            return r;
        }
        T->slot_pending[(size_t)s] = 0;
    }
    T->slot_in_use[(size_t)s] = 1;
    T->st.requests++;
    T->next_seq = q + 1;
    if (T->issued < q + 1) T->issued = q + 1;
    *dev_out = slot_ptr(T, s);
    if (resident_out) *resident_out = 0;
    prefetch(T);
    return K3MOE_OK;
}

int k3moe_trunk_release(k3moe_trunk *T, int32_t layer, k3moe_stream compute)
{
    if (!T || layer < 0 || layer >= T->M) return K3MOE_EINVAL;
    if (layer < T->P) return K3MOE_OK;
    if (T->cuda) T->cuda->compute = reinterpret_cast<cudaStream_t>(compute);
    int32_t s = -1;
    for (int32_t r = 0; r < T->R; r++)
        if (T->slot_in_use[(size_t)r] && T->slot_seq[(size_t)r] >= 0 &&
            layer_of(T, T->slot_seq[(size_t)r]) == layer &&
            (s < 0 || T->slot_seq[(size_t)r] < T->slot_seq[(size_t)s]))
            s = r;
    if (s < 0) return K3MOE_EINVAL;  // not acquired
    const int rc = T->cp.release(T->cp.ctx, T->P + s);
    T->slot_in_use[(size_t)s] = 0;
    if (rc != K3MOE_OK) return rc;
    prefetch(T);
    return K3MOE_OK;
}

int k3moe_trunk_get_stats(const k3moe_trunk *T, k3moe_trunk_stats *out)
{
    if (!T || !out) return K3MOE_EINVAL;
    *out = T->st;
    return K3MOE_OK;
}

}  // extern "C"
