// k3_policy.cpp -- host-side tooling for the expert cache's policy: offline
// replay of a recorded trace (LRU exactly as the live cache decides, and
// Belady's offline optimum), capacity sweeps for sizing, the hot set of a
// request histogram, and a trace file.
//
// The pages keep a request histogram so that a hot set can be measured and
// pinned ("kimi-k3-in-c" explainer, "The cache the project exists for"),
// size the expert cache from a recorded trace replayed offline ("Running
// Kimi K3 locally", "the four reductions"), and compare LRU with Belady over
// cache sizes ("kimi-k3-in-c: A 176 KB Engine...", "The interesting design
// decisions").  Everything here runs on the host; no CUDA call.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <exception>
#include <set>
#include <thread>
#include <unordered_map>
#include <utility>
#include <vector>

#include "k3moe.h"

namespace {

struct Trace {
    const int64_t *keys;
    const int32_t *len;
    int32_t nb;
    int64_t total;
};

// Checks a trace and returns its key count (-1 if it is not a trace).
int64_t trace_total(const int64_t *keys, const int32_t *len, int32_t nb)
{
    if (nb < 0 || (nb > 0 && !len)) return -1;
    int64_t total = 0;
    for (int32_t b = 0; b < nb; b++) {
        if (len[b] < 1) return -1;
        total += len[b];
    }
    if (total > 0 && !keys) return -1;
    for (int64_t i = 0; i < total; i++)
        if (keys[i] < 0) return -1;
    return total;
}

// LRU with the live cache's rules.  Slots are ordered for eviction by
// (last use, index); EMPTY slots by index.  Slots used by the current batch
// leave the eviction order until the batch ends, pinned slots never enter it.
int replay_lru(const Trace &t, int32_t capacity, const int64_t *pinned, int32_t npinned,
               uint8_t *hit, int64_t *hits_out)
{
    std::vector<int64_t> slot_key((size_t)capacity, -1), last((size_t)capacity, -1);
    std::vector<char> pin((size_t)capacity, 0);
    std::vector<int32_t> inb((size_t)capacity, -1);
    std::unordered_map<int64_t, int32_t> where;
    where.reserve((size_t)capacity * 2);
    std::set<int32_t> empty;
    std::set<std::pair<int64_t, int32_t>> evict;
    for (int32_t p = 0; p < npinned; p++) {
        if (!where.emplace(pinned[p], p).second) return K3MOE_EINVAL;  // a key pinned twice
        slot_key[(size_t)p] = pinned[p];
        pin[(size_t)p] = 1;
    }
    for (int32_t s = npinned; s < capacity; s++) empty.insert(s);

    int64_t hits = 0, pos = 0;
    std::vector<int32_t> batch_slots;
    std::vector<char> is_hit;
    for (int32_t b = 0; b < t.nb; b++) {
        const int32_t n = t.len[b];
        const int64_t *k = t.keys + pos;
        const int64_t now = b;
        batch_slots.clear();
        is_hit.assign((size_t)n, 0);
        auto touch = [&](int32_t s) {
            if (inb[(size_t)s] != b) {
                inb[(size_t)s] = b;
                batch_slots.push_back(s);
                if (!pin[(size_t)s]) evict.erase({last[(size_t)s], s});
            }
            last[(size_t)s] = now;
        };
        // hits first: the whole batch is needed at once
        for (int32_t i = 0; i < n; i++) {
            auto it = where.find(k[i]);
            if (it != where.end()) {
                is_hit[(size_t)i] = 1;
                touch(it->second);
            }
        }
        for (int32_t i = 0; i < n; i++) {
            if (is_hit[(size_t)i]) continue;
            auto it = where.find(k[i]);
            if (it != where.end()) {  // repeated in this batch: a hit the second time
                is_hit[(size_t)i] = 1;
                last[(size_t)it->second] = now;
                continue;
            }
            int32_t v;
            if (!empty.empty()) {
                v = *empty.begin();
                empty.erase(empty.begin());
            } else if (!evict.empty()) {
                v = evict.begin()->second;
                evict.erase(evict.begin());
                where.erase(slot_key[(size_t)v]);
            } else {
                return K3MOE_EBUSY;
            }
            slot_key[(size_t)v] = k[i];
            where[k[i]] = v;
            inb[(size_t)v] = b;
            batch_slots.push_back(v);
            last[(size_t)v] = now;
        }
        for (int32_t s : batch_slots)
            if (!pin[(size_t)s]) evict.insert({last[(size_t)s], s});
        for (int32_t i = 0; i < n; i++) {
            hits += is_hit[(size_t)i];
            if (hit) hit[pos + i] = (uint8_t)is_hit[(size_t)i];
        }
        pos += n;
    }
    *hits_out = hits;
    return K3MOE_OK;
}

// Belady: a miss evicts the resident key, not used by the current batch,
// whose next use lies farthest ahead (never used again = the end of the
// trace); equal next uses go to the lower slot.
int replay_belady(const Trace &t, int32_t capacity, uint8_t *hit, int64_t *hits_out)
{
    // next[i]: the next position holding keys[i], or total
    std::vector<int64_t> next((size_t)t.total);
    {
        std::unordered_map<int64_t, int64_t> seen;
        seen.reserve((size_t)std::min<int64_t>(t.total, 1 << 20));
        for (int64_t i = t.total - 1; i >= 0; i--) {
            auto it = seen.find(t.keys[i]);
            next[(size_t)i] = it == seen.end() ? t.total : it->second;
            seen[t.keys[i]] = i;
        }
    }
    std::vector<int64_t> slot_key((size_t)capacity, -1), nu((size_t)capacity, 0);
    std::vector<int32_t> inb((size_t)capacity, -1);
    std::unordered_map<int64_t, int32_t> where;
    where.reserve((size_t)capacity * 2);
    std::set<int32_t> empty;
    for (int32_t s = 0; s < capacity; s++) empty.insert(s);
    std::set<std::pair<int64_t, int32_t>> evict;  // (-next use, slot)

    int64_t hits = 0, pos = 0;
    std::vector<std::pair<int32_t, int64_t>> batch;  // (slot, position of its last use)
    for (int32_t b = 0; b < t.nb; b++) {
        const int32_t n = t.len[b];
        batch.clear();
        // resident keys of this batch may not be evicted while it runs
        for (int32_t i = 0; i < n; i++) {
            auto it = where.find(t.keys[pos + i]);
            if (it != where.end() && inb[(size_t)it->second] != b) {
                inb[(size_t)it->second] = b;
                evict.erase({-nu[(size_t)it->second], it->second});
            }
        }
        for (int32_t i = 0; i < n; i++) {
            const int64_t key = t.keys[pos + i];
            auto it = where.find(key);
            int32_t s;
            if (it != where.end()) {
                s = it->second;
                hits++;
                if (hit) hit[pos + i] = 1;
            } else {
                if (!empty.empty()) {
                    s = *empty.begin();
                    empty.erase(empty.begin());
                } else if (!evict.empty()) {
                    s = evict.begin()->second;
                    evict.erase(evict.begin());
                    where.erase(slot_key[(size_t)s]);
                } else {
                    return K3MOE_EBUSY;
                }
                slot_key[(size_t)s] = key;
                where[key] = s;
                inb[(size_t)s] = b;
                if (hit) hit[pos + i] = 0;
            }
            batch.push_back({s, pos + i});
        }
        // back in the eviction order, keyed by the next use after the batch
        for (const auto &sp : batch) nu[(size_t)sp.first] = next[(size_t)sp.second];
        for (const auto &sp : batch)
            if (inb[(size_t)sp.first] == b) {
                inb[(size_t)sp.first] = -1;
                evict.insert({-nu[(size_t)sp.first], sp.first});
            }
        pos += n;
    }
    *hits_out = hits;
    return K3MOE_OK;
}

int replay(const Trace &t, int32_t capacity, int32_t policy, const int64_t *pinned,
           int32_t npinned, uint8_t *hit, int64_t *hits_out)
{
    try {
        return policy == K3MOE_POLICY_LRU ? replay_lru(t, capacity, pinned, npinned, hit, hits_out)
                                          : replay_belady(t, capacity, hit, hits_out);
    } catch (const std::exception &) {
        return K3MOE_ENOMEM;
    }
}

// Runs fn(0..n-1) spread over the host's threads (fn must not throw).  A
// thread that cannot be started leaves its share to the calling thread.
template <typename Fn>
void for_each_on_threads(int32_t n, Fn &fn)
{
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    const int32_t nthreads = (int32_t)std::min<unsigned>(hw, (unsigned)n);
    std::vector<std::thread> pool;
    int32_t started = 1;  // share 0 is the calling thread's
    try {
        pool.reserve((size_t)nthreads);
        for (; started < nthreads; started++)
            pool.emplace_back([&fn, w = started, n, nthreads] {
                for (int32_t c = w; c < n; c += nthreads) fn(c);
            });
    } catch (const std::exception &) {
    }
    for (int32_t c = 0; c < n; c += nthreads) fn(c);
    for (int32_t w = started; w < nthreads; w++)
        for (int32_t c = w; c < n; c += nthreads) fn(c);
    for (auto &th : pool) th.join();
}

void put_le(unsigned char *p, uint64_t v, int bytes)
{
    for (int i = 0; i < bytes; i++) p[i] = (unsigned char)(v >> (8 * i));
}
uint64_t get_le(const unsigned char *p, int bytes)
{
    uint64_t v = 0;
    for (int i = 0; i < bytes; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}
const char kMagic[8] = {'K', '3', 'T', 'R', 'A', 'C', 'E', '1'};

}  // namespace

extern "C" {

int k3moe_trace_replay(const int64_t *keys, const int32_t *batch_len, int32_t n_batches,
                       int32_t capacity, int32_t policy, const int64_t *pinned, int32_t npinned,
                       uint8_t *hit_out, int64_t *hits_out)
{
    const int64_t total = trace_total(keys, batch_len, n_batches);
    if (total < 0 || capacity < 1 || !hits_out) return K3MOE_EINVAL;
    if (policy != K3MOE_POLICY_LRU && policy != K3MOE_POLICY_BELADY) return K3MOE_EINVAL;
    if (npinned < 0 || npinned > capacity || (npinned > 0 && !pinned)) return K3MOE_EINVAL;
    if (policy == K3MOE_POLICY_BELADY && npinned != 0) return K3MOE_EINVAL;
    for (int32_t p = 0; p < npinned; p++)
        if (pinned[p] < 0) return K3MOE_EINVAL;
    return replay({keys, batch_len, n_batches, total}, capacity, policy, pinned, npinned, hit_out,
                  hits_out);
}

int k3moe_trace_sweep(const int64_t *keys, const int32_t *batch_len, int32_t n_batches,
                      const int32_t *capacities, int32_t ncap, int32_t policy, int64_t *hits_out)
{
    const int64_t total = trace_total(keys, batch_len, n_batches);
    if (total < 0 || ncap < 1 || !capacities || !hits_out) return K3MOE_EINVAL;
    if (policy != K3MOE_POLICY_LRU && policy != K3MOE_POLICY_BELADY) return K3MOE_EINVAL;
    for (int32_t c = 0; c < ncap; c++)
        if (capacities[c] < 1) return K3MOE_EINVAL;
    const Trace t{keys, batch_len, n_batches, total};
    std::vector<int> rc;
    try {
        rc.assign((size_t)ncap, K3MOE_OK);
    } catch (const std::exception &) {
        return K3MOE_ENOMEM;
    }
    auto run = [&](int32_t c) {
        int64_t h = -1;
        const int r = replay(t, capacities[c], policy, nullptr, 0, nullptr, &h);
        hits_out[c] = r == K3MOE_OK ? h : -1;
        rc[(size_t)c] = r == K3MOE_EBUSY ? K3MOE_OK : r;
    };
    for_each_on_threads(ncap, run);
    for (int r : rc)
        if (r != K3MOE_OK) return r;
    return K3MOE_OK;
}

int k3moe_trace_pin_sweep(const int64_t *keys, const int32_t *batch_len, int32_t n_batches,
                          int32_t capacity, const int64_t *hot_keys, const int32_t *pin_counts,
                          int32_t ncounts, int64_t count_from, int64_t *hits_out)
{
    const int64_t total = trace_total(keys, batch_len, n_batches);
    if (total < 0 || capacity < 1 || ncounts < 1 || !pin_counts || !hits_out || count_from < 0)
        return K3MOE_EINVAL;
    int32_t most = 0;
    for (int32_t c = 0; c < ncounts; c++) {
        if (pin_counts[c] < 0 || pin_counts[c] > capacity) return K3MOE_EINVAL;
        most = std::max(most, pin_counts[c]);
    }
    if (most > 0 && !hot_keys) return K3MOE_EINVAL;
    for (int32_t p = 0; p < most; p++)
        if (hot_keys[p] < 0) return K3MOE_EINVAL;
    const Trace t{keys, batch_len, n_batches, total};
    std::vector<int> rc;
    try {
        rc.assign((size_t)ncounts, K3MOE_OK);
    } catch (const std::exception &) {
        return K3MOE_ENOMEM;
    }
    auto run = [&](int32_t c) {
        int64_t h = -1;
        int r = K3MOE_ENOMEM;
        try {
            std::vector<uint8_t> hit((size_t)total);
            r = replay(t, capacity, K3MOE_POLICY_LRU, hot_keys, pin_counts[c], hit.data(), &h);
            if (r == K3MOE_OK) {
                h = 0;
                for (int64_t i = count_from; i < total; i++) h += hit[(size_t)i];
            }
        } catch (const std::exception &) {
            r = K3MOE_ENOMEM;
        }
        hits_out[c] = r == K3MOE_OK ? h : -1;
        rc[(size_t)c] = r == K3MOE_EBUSY ? K3MOE_OK : r;
    };
    for_each_on_threads(ncounts, run);
    for (int r : rc)
        if (r != K3MOE_OK) return r;
    return K3MOE_OK;
}

int k3moe_hot_set(const uint32_t *hist, int64_t nkeys, int32_t n, int64_t *keys_out)
{
    if (!hist || nkeys < 1 || n < 0 || n > nkeys || (n > 0 && !keys_out)) return K3MOE_EINVAL;
    try {
        std::vector<int64_t> idx((size_t)nkeys);
        for (int64_t q = 0; q < nkeys; q++) idx[(size_t)q] = q;
        std::partial_sort(idx.begin(), idx.begin() + n, idx.end(), [&](int64_t a, int64_t b) {
            return hist[a] != hist[b] ? hist[a] > hist[b] : a < b;
        });
        std::copy(idx.begin(), idx.begin() + n, keys_out);
    } catch (const std::exception &) {
        return K3MOE_ENOMEM;
    }
    return K3MOE_OK;
}

int k3moe_trace_save(const char *path, const int64_t *keys, const int32_t *batch_len,
                     int32_t n_batches)
{
    const int64_t total = trace_total(keys, batch_len, n_batches);
    if (!path || total < 0) return K3MOE_EINVAL;
    FILE *f = fopen(path, "wb");
    if (!f) return K3MOE_EIO;
    unsigned char head[24];
    memcpy(head, kMagic, 8);
    put_le(head + 8, (uint64_t)n_batches, 8);
    put_le(head + 16, (uint64_t)total, 8);
    bool ok = fwrite(head, 1, sizeof head, f) == sizeof head;
    unsigned char buf[8];
    for (int32_t b = 0; ok && b < n_batches; b++) {
        put_le(buf, (uint32_t)batch_len[b], 4);
        ok = fwrite(buf, 1, 4, f) == 4;
    }
    for (int64_t i = 0; ok && i < total; i++) {
        put_le(buf, (uint64_t)keys[i], 8);
        ok = fwrite(buf, 1, 8, f) == 8;
    }
    if (fclose(f) != 0) ok = false;
    return ok ? K3MOE_OK : K3MOE_EIO;
}

int k3moe_trace_load(const char *path, int64_t *keys, int64_t cap_keys, int32_t *batch_len,
                     int32_t cap_batches, int64_t *n_keys, int32_t *n_batches)
{
    if (!path || !n_keys || !n_batches) return K3MOE_EINVAL;
    FILE *f = fopen(path, "rb");
    if (!f) return K3MOE_EIO;
    int rc = K3MOE_OK;
    unsigned char head[24], buf[8];
    int64_t nb = 0, nk = 0, sum = 0;
    long size = -1;
    if (fseek(f, 0, SEEK_END) == 0) size = ftell(f);
    if (size < 0 || fseek(f, 0, SEEK_SET) != 0) rc = K3MOE_EIO;
    if (rc == K3MOE_OK && (fread(head, 1, sizeof head, f) != sizeof head || memcmp(head, kMagic, 8)))
        rc = K3MOE_EINVAL;
    if (rc == K3MOE_OK) {
        nb = (int64_t)get_le(head + 8, 8);
        nk = (int64_t)get_le(head + 16, 8);
        // the sizes must describe exactly the rest of the file
        if (nb < 0 || nb > INT32_MAX || nk < 0 || nk > (int64_t)1 << 40 ||
            (int64_t)sizeof head + 4 * nb + 8 * nk != (int64_t)size)
            rc = K3MOE_EINVAL;
    }
    if (rc == K3MOE_OK) {
        *n_batches = (int32_t)nb;
        *n_keys = nk;
        if ((batch_len && cap_batches < nb) || (keys && cap_keys < nk)) rc = K3MOE_EINVAL;
    }
    for (int64_t b = 0; rc == K3MOE_OK && b < nb; b++) {
        if (fread(buf, 1, 4, f) != 4) {
            rc = K3MOE_EIO;
            break;
        }
        const int32_t l = (int32_t)(uint32_t)get_le(buf, 4);
        if (l < 1) rc = K3MOE_EINVAL;
        sum += l;
        if (batch_len) batch_len[b] = l;
    }
    if (rc == K3MOE_OK && sum != nk) rc = K3MOE_EINVAL;
    for (int64_t i = 0; rc == K3MOE_OK && keys && i < nk; i++) {
        if (fread(buf, 1, 8, f) != 8) {
            rc = K3MOE_EIO;
            break;
        }
        keys[i] = (int64_t)get_le(buf, 8);
        if (keys[i] < 0) rc = K3MOE_EINVAL;
    }
    fclose(f);
    return rc;
}

}  // extern "C"
