"""Host logic of the expert cache, driven through the C ABI with a fake
copier (no GPU): replacement decisions against the oracle's LRU replay, the
pages' cyclic-scan results, the INFLIGHT regression, refusals and injected
copy failures."""
import ctypes

import numpy as np
import pytest

import oracle
from mxfp4_routed_expert_select_gb300 import k3moe as k

EB = 64  # bytes per fake expert blob


class FakeCopier:
    """Host arena + memcpy; records every copy; can fail the n-th copy."""

    def __init__(self, fail_on=()):
        self.copies = []
        self.waits = []
        self.releases = []
        self.fail_on = set(fail_on)
        self.arena = None

        def alloc(ctx, nbytes, out):
            self.arena = ctypes.create_string_buffer(nbytes)
            out[0] = ctypes.addressof(self.arena)
            return 0

        def free(ctx, p):
            return 0

        def copy(ctx, slot, dst, src, nbytes):
            n = len(self.copies)
            self.copies.append((slot, dst, src))
            if n in self.fail_on:
                return k.K3MOE_ECUDA
            ctypes.memmove(dst, src, nbytes)
            return 0

        def wait(ctx, slot):
            self.waits.append(slot)
            return 0

        def release(ctx, slot):
            self.releases.append(slot)
            return 0
        self._fns = (k.ALLOC_FN(alloc), k.FREE_FN(free), k.COPY_FN(copy), k.SLOT_FN(wait),
                     k.SLOT_FN(release))
        self.struct = k.Copier(None, *self._fns)


def make_cache(n_layers, n_experts, slots, copier=None):
    nkeys = n_layers * n_experts
    host = [ctypes.create_string_buffer(bytes([q % 251]) * EB) for q in range(nkeys)]
    ptrs = [ctypes.addressof(b) for b in host]
    cp = copier or FakeCopier()
    c = k.Cache(slots * EB + EB // 2, EB, ptrs, n_layers, n_experts, copier=cp.struct)
    c._host = host
    return c, cp


def run_trace(c, batches):
    hits = []
    for b in batches:
        ptrs, hit, st = c.acquire(b)
        assert st == 0
        for key, p in zip(b, ptrs):  # the slot holds this key's bytes
            assert ctypes.string_at(p, 1)[0] == key % 251
        hits.extend(hit.tolist())
        c.release()
    return np.array(hits, np.uint8)


def test_cyclic_scan_lru_hits_zero_and_pinned_prefix(golden):
    """LRU of 90 slots over a 93-key cycle hits 0; pinning 90 keys with one
    ring slot hits 90/93 ("kimi-k3-in-c: A 176 KB Engine...", 'The interesting
    design decisions')."""
    M, C = 93, 90
    c, _ = make_cache(1, M, C)
    hits = run_trace(c, [[q] for q in list(range(M)) * 4])
    assert hits.sum() == 0
    c, _ = make_cache(1, M, C + 1)
    for q in range(C):
        assert c.pin(q) == 0
    hits = run_trace(c, [[q] for q in list(range(M)) * 4])
    assert hits.sum() == C * 4
    assert round(100 * hits.sum() / hits.size, 1) == golden["trunk_cycle_pinned"]["hit_rate_pct"]
    assert c.stats()["pinned"] == C


@pytest.mark.parametrize("slots,seed", [(16, 0), (24, 1), (40, 2), (100, 3)])
def test_replacement_matches_oracle_lru(slots, seed):
    """Zipf-biased batches of 16 distinct experts over 2 layers: the hit/miss
    sequence equals the oracle's replay exactly."""
    rng = np.random.default_rng(seed)
    L, E = 2, 64
    p = np.arange(1, E + 1) ** -1.1
    p /= p.sum()
    batches = []
    for t in range(60):
        for l in range(L):
            ex = np.sort(rng.choice(E, 16, replace=False, p=p))
            batches.append(list(l * E + ex))
    c, cp = make_cache(L, E, slots)
    hits = run_trace(c, batches)
    keys = np.concatenate(batches)
    ref_hits, ref = oracle.cache_lru(keys, np.full(len(batches), 16, np.int32), slots)
    assert ref_hits >= 0
    assert np.array_equal(hits, ref)
    st = c.stats()
    assert st["hits"] == ref_hits and st["misses"] == keys.size - ref_hits
    assert st["h2d_bytes"] == st["misses"] * EB and st["hbm_bytes"] == keys.size * EB
    hist = c.histogram()
    assert np.array_equal(hist, np.bincount(keys, minlength=L * E))


def test_batch_misses_get_distinct_slots():
    """The explainer page's bug: a batch prefetch handed the same slot to
    several reads.  Every miss of one batch must get its own slot, also when
    the cache starts full and every victim comes from the LRU scan."""
    c, cp = make_cache(1, 64, 16)
    run_trace(c, [list(range(16))])
    n0 = len(cp.copies)
    ptrs, hit, st = c.acquire(list(range(16, 32)))
    new = cp.copies[n0:]
    assert len(new) == 16 and len({s for s, _, _ in new}) == 16
    assert len(set(ptrs)) == 16
    assert c.stats()["inflight"] == 0
    c.release()


def test_in_use_slots_are_not_evicted_and_busy_is_refused():
    c, cp = make_cache(1, 64, 8)
    ptrs, hit, st = c.acquire(list(range(8)))
    # without a release all 8 slots are in use: a new key cannot be placed
    _, _, st = c.acquire([9], raise_on_error=False)
    assert st == k.K3MOE_EBUSY
    assert c.stats()["lookups"] == 8  # the refused call changed nothing
    c.release()
    _, hit, st = c.acquire([9])
    assert st == 0 and hit[0] == 0
    c.release()


def test_injected_copy_failure_leaves_key_uncached():
    cp = FakeCopier(fail_on={2})
    c, _ = make_cache(1, 32, 8, copier=cp)
    ptrs, hit, st = c.acquire([0, 1, 2, 3], raise_on_error=False)
    assert st == k.K3MOE_ECUDA
    assert c.slot_of(2) == -1 and c.slot_of(0) >= 0 and c.slot_of(3) >= 0
    c.release()
    ptrs, hit, st = c.acquire([2, 0])
    assert st == 0 and list(hit) == [0, 1]
    assert ctypes.string_at(ptrs[0], 1)[0] == 2
    c.release()


def test_refusals():
    host = [ctypes.create_string_buffer(EB) for _ in range(4)]
    ptrs = [ctypes.addressof(b) for b in host]
    cp = FakeCopier()
    with pytest.raises(k.K3Error) as ei:
        k.Cache(EB - 1, EB, ptrs, 1, 4, copier=cp.struct)  # less than one slot
    assert ei.value.status == k.K3MOE_EINVAL
    c = k.Cache(2 * EB, EB, ptrs, 1, 4, copier=cp.struct)
    _, _, st = c.acquire([4], raise_on_error=False)
    assert st == k.K3MOE_EINVAL
    assert c.pin(7) == k.K3MOE_EINVAL


def test_split_acquire_defers_the_waits_and_keeps_the_plan():
    """k3moe_cache_acquire_split: the same slots, copies and counters as the
    plain acquire, but the misses' waits come only with wait_copies (or with
    the next acquire / release), and until then their keys are INFLIGHT."""
    ca, cpa = make_cache(1, 64, 8)
    cb, cpb = make_cache(1, 64, 8)
    batches = [[0, 1, 2, 3], [2, 3, 4, 5], [6, 7, 8, 9], [0, 9, 10, 11]]
    for b in batches:
        pa, ha, _ = ca.acquire(b)
        nw = len(cpb.waits)
        pb, hb, _ = cb.acquire(b, split=True)
        misses = int((hb == 0).sum())
        assert len(cpb.waits) == nw  # no wait yet
        assert cb.stats()["inflight"] == misses
        for key, h in zip(b, hb):
            assert (cb.slot_of(key) >= 0) == bool(h)
        assert cb.wait_copies() == 0
        assert len(cpb.waits) == nw + misses
        assert cb.stats()["inflight"] == 0
        assert list(ha) == list(hb)
        assert [ca.slot_of(x) for x in b] == [cb.slot_of(x) for x in b]
        for key, p in zip(b, pb):
            assert ctypes.string_at(p, 1)[0] == key % 251
        ca.release()
        cb.release()
    assert [s for s, _, _ in cpa.copies] == [s for s, _, _ in cpb.copies]
    assert cpa.waits == cpb.waits
    assert ca.stats() == cb.stats()


def test_release_and_the_next_acquire_wait_for_pending_copies():
    c, cp = make_cache(1, 64, 8)
    _, hit, _ = c.acquire([0, 1, 2], split=True)
    assert cp.waits == [] and c.stats()["inflight"] == 3
    c.release()  # publishes before marking the slots free
    assert sorted(cp.waits) == sorted(s for s, _, _ in cp.copies)
    assert len(cp.releases) == 3 and c.stats()["inflight"] == 0
    _, _, _ = c.acquire([3], split=True)
    # a second split acquire of the pending key finds it as a hit, not a miss
    _, hit, _ = c.acquire([3, 0], split=True)
    assert list(hit) == [1, 1] and len(cp.copies) == 4
    assert c.stats()["inflight"] == 0
    c.release()


def test_wait_copy_waits_for_one_slot():
    c, cp = make_cache(1, 64, 8)
    c.acquire([0, 1])
    c.release()
    ptrs, hit, _ = c.acquire([0, 5, 6], split=True)
    assert list(hit) == [1, 0, 0] and cp.waits == [cp.copies[0][0], cp.copies[1][0]]
    n0 = len(cp.waits)
    assert c.wait_copy(ptrs[0]) == 0 and len(cp.waits) == n0  # a hit: nothing to wait for
    assert c.wait_copy(ptrs[2]) == 0
    assert cp.waits[n0:] == [c.slot_of(6)] and c.slot_of(5) == -1
    assert c.stats()["inflight"] == 1
    assert c.wait_copy(ptrs[2]) == 0 and len(cp.waits) == n0 + 1  # already waited for
    assert c.wait_copy(ptrs[1] + 1) == k.K3MOE_EINVAL  # not a slot start
    assert c.wait_copy(ptrs[1]) == 0 and c.slot_of(5) >= 0
    assert c.stats()["inflight"] == 0
    c.release()
