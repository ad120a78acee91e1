"""Pins of the oracle's cache replay (LRU with pinning, Belady) against the
pages' cyclic-scan results and brute force (no GPU)."""
import itertools

import numpy as np

import oracle


def test_lru_over_cycle_longer_than_capacity_hits_zero(golden):
    """An LRU of 90 slots over a 93-layer cycle hits exactly zero
    ("kimi-k3-in-c: A 176 KB Engine...", 'The interesting design decisions')."""
    g = golden["trunk_cycle_lru"]
    M, C = g["layers"], g["slots"]
    keys = np.tile(np.arange(M), 5)
    hits, hit = oracle.cache_lru(keys, np.ones(keys.size, np.int32), C)
    assert hits == 0 and hits / keys.size == g["hit_rate"]


def test_pinned_prefix_hits_n_over_m(golden):
    """Pinning the first N layers of an M-layer cycle (plus one ring slot)
    hits N/M: 96.8% at N = 90 of 93 (same section)."""
    g = golden["trunk_cycle_pinned"]
    M, N = g["layers"], g["pinned"]
    cycles = 4
    keys = np.tile(np.arange(M), cycles)
    hits, hit = oracle.cache_lru(keys, np.ones(keys.size, np.int32), N + 1, pinned=np.arange(N))
    assert hits == N * cycles
    assert round(100 * hits / keys.size, 1) == g["hit_rate_pct"]


def test_batch_keys_never_evict_each_other():
    """A batch (one token's experts at one layer) must be resident at once:
    with capacity == batch size, every new batch misses entirely and no key of
    the current batch is evicted by another of the same batch."""
    keys = np.array([1, 2, 3, 4, 1, 2, 5, 6, 5, 6, 1, 2])
    bl = np.array([4, 4, 4], np.int32)
    hits, hit = oracle.cache_lru(keys, bl, 4)
    # batch 2: 1,2 hit; 5,6 evict 3,4 (LRU, not in batch)
    # batch 3: 5,6 hit; 1,2 hit
    assert list(hit) == [0, 0, 0, 0, 1, 1, 0, 0, 1, 1, 1, 1]
    assert hits == 6
    assert oracle.cache_lru(keys, bl, 3)[0] == -1  # cannot place a batch of 4


def _brute_lru(keys, bl, C):
    """Straight list-based LRU used as an independent replay."""
    order = []  # least recent first
    hits = 0
    pos = 0
    for n in bl:
        batch = list(keys[pos:pos + n])
        for k in batch:
            if k in order:
                hits += 1
                order.remove(k)
                order.append(k)
            else:
                if len(order) >= C:
                    for v in order:
                        if v not in batch:
                            order.remove(v)
                            break
                order.append(k)
        pos += n
    return hits


def _brute_belady(keys, bl, C):
    """Offline optimum by exhaustive search over eviction choices (tiny)."""
    keys = list(keys)
    bounds = list(itertools.accumulate([0] + list(bl)))

    def rec(i, cache):
        if i == len(keys):
            return 0
        b = max(j for j in range(len(bl)) if bounds[j] <= i)
        batch = keys[bounds[b]:bounds[b + 1]]
        k = keys[i]
        if k in cache:
            return 1 + rec(i + 1, cache)
        if len(cache) < C:
            return rec(i + 1, cache | {k})
        best = -1
        for v in cache:
            if v in batch:
                continue
            best = max(best, rec(i + 1, (cache - {v}) | {k}))
        return best
    return rec(0, frozenset())


def test_lru_and_belady_against_brute_force():
    rng = np.random.default_rng(12)
    for trial in range(30):
        n = int(rng.integers(6, 14))
        keys = rng.integers(0, 6, n)
        bl = np.ones(n, np.int32)
        C = int(rng.integers(1, 4))
        assert oracle.cache_lru(keys, bl, C)[0] == _brute_lru(keys, bl, C)
        assert oracle.cache_belady(keys, bl, C) == _brute_belady(keys, bl, C)
    # batched traces of distinct keys per batch
    for trial in range(20):
        nb = int(rng.integers(2, 6))
        batches = [rng.choice(8, 2, replace=False) for _ in range(nb)]
        keys = np.concatenate(batches)
        bl = np.full(nb, 2, np.int32)
        C = int(rng.integers(2, 5))
        assert oracle.cache_lru(keys, bl, C)[0] == _brute_lru(keys, bl, C)
        assert oracle.cache_belady(keys, bl, C) == _brute_belady(keys, bl, C)


def test_belady_at_least_lru_on_zipf_trace():
    rng = np.random.default_rng(1)
    ranks = np.arange(1, 201)
    p = ranks ** -1.1
    p /= p.sum()
    batches = [rng.choice(200, 16, replace=False, p=p) for _ in range(200)]
    keys = np.concatenate(batches)
    bl = np.full(len(batches), 16, np.int32)
    for C in [16, 32, 64]:
        lru = oracle.cache_lru(keys, bl, C)[0]
        bel = oracle.cache_belady(keys, bl, C)
        assert 0 <= lru <= bel <= keys.size
