"""Cache policy tooling of the library (host-side, no GPU): offline replay of
a recorded trace against the oracle's LRU and Belady replays, the live cache
against its own replayed trace, the pages' cyclic-scan numbers, hot sets from
the request histogram, capacity sweeps and the trace file.

The pages keep a request histogram so that a hot set can be measured and
pinned ("kimi-k3-in-c" explainer, "The cache the project exists for"), size
the expert cache from a recorded trace ("Running Kimi K3 locally", the four
reductions) and compare LRU with Belady over sizes ("kimi-k3-in-c: A 176 KB
Engine...", "The interesting design decisions")."""
import ctypes
import os

import numpy as np
import pytest

import oracle
import synth
from mxfp4_routed_expert_select_gb300 import k3moe as k
from test_cache_host import FakeCopier, make_cache, run_trace


def _random_trace(rng, dup):
    nb = int(rng.integers(1, 40))
    bs = int(rng.integers(1, 6))
    space = int(rng.integers(bs, 30))
    batches = [rng.choice(space, bs, replace=dup) for _ in range(nb)]
    return np.concatenate(batches).astype(np.int64), np.full(nb, bs, np.int32), space


@pytest.mark.parametrize("dup", [False, True])
def test_lru_replay_matches_the_oracle_decision_for_decision(dup):
    rng = np.random.default_rng(21 + dup)
    busy = 0
    for _ in range(150):
        keys, bl, space = _random_trace(rng, dup)
        C = int(rng.integers(1, 20))
        npin = int(rng.integers(0, min(C, space) + 1)) if rng.integers(0, 2) else 0
        pinned = rng.choice(space, npin, replace=False)
        ref_hits, ref = oracle.cache_lru(keys, bl, C, pinned=pinned)
        hits, hit = k.trace_replay(keys, bl, C, "lru", pinned)
        assert hits == ref_hits
        if ref_hits >= 0:
            assert np.array_equal(hit, ref)
        busy += ref_hits < 0
    assert 0 < busy < 150  # both outcomes were exercised


def test_belady_replay_matches_the_oracle():
    rng = np.random.default_rng(5)
    for dup in (False, True):
        for _ in range(150):
            keys, bl, _ = _random_trace(rng, dup)
            C = int(rng.integers(1, 20))
            assert k.trace_replay(keys, bl, C, "belady")[0] == oracle.cache_belady(keys, bl, C)


def test_replay_of_the_pages_cyclic_scan(golden):
    """LRU of 90 slots over a 93-layer cycle hits zero; pinning the first 90
    (one ring slot left) hits 90/93 = 96.8% ("kimi-k3-in-c: A 176 KB
    Engine...", 'The interesting design decisions')."""
    g = golden["trunk_cycle_lru"]
    keys = np.tile(np.arange(g["layers"]), 6)
    bl = np.ones(keys.size, np.int32)
    assert k.trace_replay(keys, bl, g["slots"])[0] == 0
    g = golden["trunk_cycle_pinned"]
    M, N = g["layers"], g["pinned"]
    keys = np.tile(np.arange(M), 6)
    hits, _ = k.trace_replay(keys, np.ones(keys.size, np.int32), N + 1, "lru", np.arange(N))
    assert hits == 6 * N and round(100 * hits / keys.size, 1) == g["hit_rate_pct"]
    # a cycle of M distinct keys with C < M slots misses at least M - C times
    # per cycle (at most C of them are resident when it starts); the offline
    # optimum reaches that bound after the cold first cycle
    for C in (N, N + 1, 50):
        assert k.trace_replay(keys, np.ones(keys.size, np.int32), C, "belady")[0] == 5 * C


def test_live_cache_records_a_trace_its_replay_reproduces():
    """The recorded trace of a live cache, replayed offline under LRU, gives
    the live cache's own hit flags, with and without keys pinned first."""
    rng = np.random.default_rng(9)
    for pinned in ([], [3, 17, 40]):
        c, cp = make_cache(3, 16, 20)
        for key in pinned:
            assert c.pin(key) == 0
        c.record_trace(True)
        batches = [rng.choice(48, int(rng.integers(1, 9)), replace=False) for _ in range(300)]
        hits = run_trace(c, batches)
        keys, bl = c.trace()
        assert np.array_equal(keys, np.concatenate(batches))
        assert np.array_equal(bl, [len(b) for b in batches])
        n, flags = k.trace_replay(keys, bl, 20, "lru", pinned)
        assert np.array_equal(flags, hits) and n == hits.sum()
        c.close()


def test_trace_record_skips_pins_and_refused_batches_and_restarts_clean():
    c, _ = make_cache(1, 8, 3)
    c.record_trace(True)
    assert c.pin(5) == 0  # not a request
    run_trace(c, [[1], [2, 3]])  # 2 and 3 take the free slot and 1's
    # 2 and 3 hit, 1 finds only the pinned slot and the batch's own: refused
    ptrs, hit, st = c.acquire([1, 2, 3], raise_on_error=False)
    assert st == k.K3MOE_EBUSY
    keys, bl = c.trace()
    assert keys.tolist() == [1, 2, 3] and bl.tolist() == [1, 2]
    c.record_trace(False)
    run_trace(c, [[4]])
    assert c.trace()[0].tolist() == [1, 2, 3]
    c.record_trace(True)
    assert c.trace()[0].size == 0
    c.close()


def test_request_histogram_has_the_pages_size(golden):
    """One counter per (MoE layer, expert) key: 92 x 896 = 82,432 counters of
    4 bytes, 330 KB (the explainer page, 'The cache the project exists
    for'), counting every request."""
    g = golden["request_histogram"]
    buf = ctypes.create_string_buffer(64)
    n = g["layers"] * g["experts_per_layer"]
    cp = FakeCopier()
    c = k.Cache(4 * 64, 64, [ctypes.addressof(buf)] * n, g["layers"], g["experts_per_layer"],
                copier=cp.struct)
    h = c.histogram()
    assert h.size == g["counters"] and round(h.nbytes / 1000) == g["kb"]
    for keys in ([5, 82431], [5], [7, 5]):
        c.acquire(keys)
        c.release()
    h = c.histogram()
    assert (h[5], h[7], h[82431], int(h.sum())) == (3, 1, 1, 5)
    c.close()


def test_hot_set_is_the_most_requested_keys_ties_to_the_lower_key():
    rng = np.random.default_rng(2)
    hist = rng.integers(0, 5, 300).astype(np.uint32)  # many ties
    want = sorted(range(hist.size), key=lambda q: (-int(hist[q]), q))
    for n in (0, 1, 7, 150, 300):
        assert k.hot_set(hist, n).tolist() == want[:n]
    with pytest.raises(k.K3Error):
        k.hot_set(hist, 301)


def test_pin_hot_uses_the_cache_histogram_and_unpin_releases():
    c, _ = make_cache(1, 10, 4)
    run_trace(c, [[7], [7, 2], [7, 2, 9], [1]])
    assert c.pin_hot(2) == 0
    s7, s2 = c.slot_of(7), c.slot_of(2)
    assert s7 >= 0 and s2 >= 0 and c.stats()["pinned"] == 2
    run_trace(c, [[3, 4], [5, 6]])  # two free slots churn; 7 and 2 stay
    assert c.slot_of(7) == s7 and c.slot_of(2) == s2
    c.unpin(7)
    assert c.stats()["pinned"] == 1
    run_trace(c, [[3, 4], [5, 6], [8, 0]])
    assert c.slot_of(7) == -1 and c.slot_of(2) == s2
    # counts now 7:3, then 2, 3, 4, 5, 6 at 2 each: the top 4 are 7, 2, 3, 4
    assert c.pin_hot(4) == 0 and c.stats()["pinned"] == 4
    assert sorted(c.slot_of(q) for q in (7, 2, 3, 4)) == [0, 1, 2, 3]
    assert c.acquire([9], raise_on_error=False)[2] == k.K3MOE_EBUSY  # every slot pinned
    assert c.pin_hot(5) == k.K3MOE_EBUSY
    c.close()


def test_sweep_equals_one_replay_per_capacity():
    rng = np.random.default_rng(4)
    ranks = np.arange(1, 201)
    p = ranks ** -1.1
    p /= p.sum()
    batches = [rng.choice(200, 8, replace=False, p=p) for _ in range(300)]
    keys, bl = np.concatenate(batches), np.full(300, 8, np.int32)
    caps = np.array([4, 8, 9, 16, 33, 64, 100, 200, 250])
    for pol in ("lru", "belady"):
        sw = k.trace_sweep(keys, bl, caps, pol)
        for cap, h in zip(caps, sw):
            assert h == k.trace_replay(keys, bl, cap, pol)[0]
        assert sw[0] == -1  # a batch of 8 cannot be placed in 4 slots
    lru, bel = k.trace_sweep(keys, bl, caps, "lru"), k.trace_sweep(keys, bl, caps, "belady")
    assert np.all(lru[1:] <= bel[1:])
    # with room for every key, only the first request of each key misses
    assert lru[-1] == bel[-1] == keys.size - np.unique(keys).size


def _routing_trace(T, L=4, E=896, K=16, pool=4):
    """Decode-order keys (layer * E + expert) of T tokens through L layers:
    logits ~ N(0, (0.02 sqrt 7168)^2), the spread of a unit-RMS token through
    a bf16 router of std 0.02, plus each layer's Zipf(1.1) selection bias;
    top-K by the oracle."""
    ids = np.zeros((T, L, K), np.int64)
    for l in range(L):
        lg = synth.normal_f64((T, E), synth.tag(synth.K_MISC, pool, l, 7), std=0.02 * np.sqrt(7168))
        bias = np.asarray(synth.bias_zipf(pool, l, E), np.float64)
        ids[:, l] = oracle.topk(lg, K, bias)[0]
    keys = (ids + (np.arange(L) * E)[None, :, None]).reshape(-1)
    return keys, np.full(T * L, K, np.int32)


def test_pinning_the_measured_hot_set_beats_plain_lru_on_a_zipf_trace():
    """4 layers x 896 experts behind 455 slots, top-16 per token and layer:
    pin the hottest keys of the first half's request histogram, leave one
    batch of slots to LRU, and the second half hits more often than under
    plain LRU; Belady's offline optimum stays above both."""
    keys, bl = _routing_trace(512)
    C, half = 455, keys.size // 2
    hist = np.bincount(keys[:half], minlength=4 * 896).astype(np.uint32)
    hot = k.hot_set(hist, C - 16)
    lru_hits, lru = k.trace_replay(keys, bl, C)
    pin_hits, pin = k.trace_replay(keys, bl, C, "lru", hot)
    assert (pin_hits, pin.tolist()) == (lambda r: (r[0], r[1].tolist()))(
        oracle.cache_lru(keys, bl, C, pinned=hot))
    bel = k.trace_replay(keys, bl, C, "belady")[1]
    r_lru, r_pin, r_bel = lru[half:].mean(), pin[half:].mean(), bel[half:].mean()
    assert r_pin > r_lru + 0.03, (r_lru, r_pin)
    assert r_bel > r_pin

    # the same through a live cache: record, pin the measured hot set, go on
    c, _ = make_cache(4, 896, C)
    c.record_trace(True)
    first = run_trace(c, np.split(keys[:half], half // 16))
    assert np.array_equal(first, lru[:half])
    assert np.array_equal(c.histogram(), hist)
    assert c.pin_hot(C - 16) == 0
    second = run_trace(c, np.split(keys[half:], half // 16))
    assert second.mean() > r_lru + 0.03
    c.close()


def test_pin_sweep_equals_replays_and_finds_a_better_hot_set():
    """Each pin count's hits (counted from the second half) equal those of a
    replay with that many hot keys pinned; on the Zipf trace some pinned hot
    set beats plain LRU (0 pinned) on the held-out half."""
    keys, bl = _routing_trace(256)
    C, half = 455, keys.size // 2
    hot = k.hot_set(np.bincount(keys[:half], minlength=4 * 896).astype(np.uint32), C)
    counts = [0, 64, 200, 350, C - 16, C - 15, C]
    sw = k.trace_pin_sweep(keys, bl, C, hot, counts, count_from=half)
    for n, h in zip(counts, sw):
        hits, flags = k.trace_replay(keys, bl, C, "lru", hot[:n])
        assert h == (-1 if hits < 0 else int(flags[half:].sum()))
    assert sw[-1] == -1  # every slot pinned: the first unpinned request finds no slot
    assert max(sw[1:5]) > sw[0]
    with pytest.raises(k.K3Error):
        k.trace_pin_sweep(keys, bl, C, hot, [C + 1])


def test_trace_file_round_trip_and_refusals(tmp_path):
    keys, bl = _routing_trace(8)
    path = str(tmp_path / "t.k3trace")
    k.trace_save(path, keys, bl)
    assert os.path.getsize(path) == 24 + 4 * bl.size + 8 * keys.size
    k2, b2 = k.trace_load(path)
    assert np.array_equal(k2, keys) and np.array_equal(b2, bl)
    raw = open(path, "rb").read()
    lib = k.lib()
    nk, nb = ctypes.c_int64(), ctypes.c_int32()

    def load_status(data):
        p = str(tmp_path / "bad")
        with open(p, "wb") as fh:
            fh.write(data)
        return lib.k3moe_trace_load(p.encode(), None, 0, None, 0, ctypes.byref(nk), ctypes.byref(nb))
    assert load_status(raw) == 0
    assert load_status(raw[:-1]) == k.K3MOE_EINVAL  # truncated
    assert load_status(b"K3TRACE2" + raw[8:]) == k.K3MOE_EINVAL  # not this format
    bad_len = bytearray(raw)
    bad_len[24:28] = (0).to_bytes(4, "little")  # an empty batch
    full = np.zeros(keys.size, np.int64)
    p = str(tmp_path / "bad2")
    open(p, "wb").write(bytes(bad_len))
    assert lib.k3moe_trace_load(p.encode(), full.ctypes.data, full.size, None, 0, ctypes.byref(nk),
                                ctypes.byref(nb)) == k.K3MOE_EINVAL
    assert lib.k3moe_trace_load(str(tmp_path / "missing").encode(), None, 0, None, 0,
                                ctypes.byref(nk), ctypes.byref(nb)) == k.K3MOE_EIO
    small = np.zeros(keys.size - 1, np.int64)
    assert lib.k3moe_trace_load(path.encode(), small.ctypes.data, small.size, None, 0,
                                ctypes.byref(nk), ctypes.byref(nb)) == k.K3MOE_EINVAL


def test_replay_refusals():
    lib = k.lib()
    keys = np.array([1, 2, 3], np.int64)
    bl = np.array([2, 1], np.int32)
    h = ctypes.c_int64()

    def st(keys=keys, bl=bl, cap=4, pol=k.K3MOE_POLICY_LRU, pin=None, npin=0):
        return lib.k3moe_trace_replay(keys.ctypes.data, bl.ctypes.data, bl.size, cap, pol,
                                      None if pin is None else pin.ctypes.data, npin, None,
                                      ctypes.byref(h))
    assert st() == 0 and h.value == 0
    assert st(keys=np.array([1, -2, 3], np.int64)) == k.K3MOE_EINVAL
    assert st(bl=np.array([3, 0], np.int32)) == k.K3MOE_EINVAL
    assert st(cap=0) == k.K3MOE_EINVAL
    assert st(pol=2) == k.K3MOE_EINVAL
    assert st(pin=np.array([1, 2], np.int64), npin=2, cap=1) == k.K3MOE_EINVAL
    assert st(pin=np.array([1], np.int64), npin=1, pol=k.K3MOE_POLICY_BELADY) == k.K3MOE_EINVAL
    assert st(pin=np.array([5, 5], np.int64), npin=2) == k.K3MOE_EINVAL  # pinned twice
    assert st(cap=1) == k.K3MOE_EBUSY  # a batch of 2 in one slot
