"""Host logic of the dense-trunk streamer (resident prefix + ring slots),
driven through the C ABI with a logging fake copier (no GPU): the pages'
cyclic-scan numbers, bytes per token, prefetch overlap, slot reuse only
after release, out-of-order requests and refusals."""
import ctypes

import numpy as np
import pytest

from mxfp4_routed_expert_select_gb300 import k3moe as k


class LogCopier:
    """Host arena + memcpy; one log of every copier call in order."""

    def __init__(self, fail_on=()):
        self.log = []
        self.arena = None
        self.fail_on = set(fail_on)
        self.ncopy = 0

        def alloc(ctx, nbytes, out):
            self.arena = ctypes.create_string_buffer(nbytes)
            out[0] = ctypes.addressof(self.arena)
            return 0

        def free(ctx, p):
            return 0

        def copy(ctx, slot, dst, src, nbytes):
            n = self.ncopy
            self.ncopy += 1
            self.log.append(("copy", slot, src))
            if n in self.fail_on:
                return k.K3MOE_ECUDA
            ctypes.memmove(dst, src, nbytes)
            return 0

        def wait(ctx, slot):
            self.log.append(("wait", slot, None))
            return 0

        def release(ctx, slot):
            self.log.append(("release", slot, None))
            return 0
        self._fns = (k.ALLOC_FN(alloc), k.FREE_FN(free), k.COPY_FN(copy), k.SLOT_FN(wait),
                     k.SLOT_FN(release))
        self.struct = k.Copier(None, *self._fns)


def make_trunk(sizes, pinned_bytes, ring, copier=None):
    host = [ctypes.create_string_buffer(bytes([(7 * l + 3) % 251]) * n) for l, n in enumerate(sizes)]
    cp = copier or LogCopier()
    t = k.Trunk([ctypes.addressof(b) for b in host], sizes, pinned_bytes, ring, copier=cp.struct)
    t._host = host
    return t, cp


def walk(t, M, tokens, release=True):
    """Tokens through layers 0..M-1; checks every layer's bytes."""
    res = []
    for _ in range(tokens):
        for l in range(M):
            p, r, st = t.acquire(l)
            assert ctypes.string_at(p, 1)[0] == (7 * l + 3) % 251
            res.append(r)
            if release:
                assert t.release(l) == 0
    return np.array(res)


def test_pinned_prefix_hits_n_over_m_on_the_pages_cycle(golden):
    """93 layers, a prefix budget of 90 layers, one ring slot: 90/93 = 96.8%
    of requests are resident ("kimi-k3-in-c: A 176 KB Engine...", 'The
    interesting design decisions'), and every token copies exactly the 3
    streamed layers once."""
    g = golden["trunk_cycle_pinned"]
    M, N, B = g["layers"], g["pinned"], 1024
    t, cp = make_trunk([B] * M, N * B, 1)
    st0 = t.stats()
    assert st0["pinned_layers"] == N and st0["h2d_bytes"] == N * B
    res = walk(t, M, 5)
    assert res.sum() == 5 * N and round(100 * res.mean(), 1) == g["hit_rate_pct"]
    assert t.stats()["h2d_bytes"] - st0["h2d_bytes"] == 5 * (M - N) * B
    t.close()


@pytest.mark.parametrize("ring", [1, 2, 3, 5])
def test_ring_prefetches_and_reuses_a_slot_only_after_its_release(ring):
    sizes = [512, 1024, 256, 768, 1024, 512, 256]
    M = len(sizes)
    t, cp = make_trunk(sizes, 512 + 1024, ring)  # layers 0 and 1 resident
    P = t.stats()["pinned_layers"]
    assert P == 2
    res = walk(t, M, 4)
    st = t.stats()
    S = M - P
    assert res.sum() == 4 * P
    # every streamed layer was copied once per token (plus the window ahead)
    streamed_copies = [e for e in cp.log if e[0] == "copy" and e[1] >= P]
    assert 4 * S <= len(streamed_copies) <= 4 * S + ring - 1
    assert st["h2d_bytes"] == sum(sizes[:P]) + sum(sizes[P + (i % S)] for i in range(len(streamed_copies)))
    # with two or more slots every streamed acquire after the first found its
    # copy already issued, i.e. it overlapped the previous layer's compute
    assert st["prefetched"] == (4 * S if ring >= 2 else 0)
    # a slot is copied into again only after its previous layer's release
    busy = {}
    for kind, slot, _ in cp.log:
        if slot < P:
            continue
        if kind == "copy":
            assert not busy.get(slot, False), cp.log
            busy[slot] = "copied"
        elif kind == "wait":
            busy[slot] = True
        elif kind == "release":
            busy[slot] = False
    t.close()


def test_everything_resident_needs_no_ring():
    t, cp = make_trunk([256] * 4, 4 * 256, 0)
    assert t.stats()["pinned_layers"] == 4 and t.stats()["ring_slots"] == 0
    assert walk(t, 4, 3).all()
    assert [e[0] for e in cp.log].count("copy") == 4
    t.close()


def test_out_of_order_requests_are_served():
    sizes = [256] * 6
    t, cp = make_trunk(sizes, 256, 2)  # layer 0 resident, 1..5 streamed
    for l in [3, 1, 5, 5, 2, 0, 4, 1]:
        p, r, st = t.acquire(l)
        assert ctypes.string_at(p, 1)[0] == (7 * l + 3) % 251
        assert r == (l == 0)
        assert t.release(l) == 0
    t.close()


def test_holding_every_slot_refuses_the_next_layer():
    t, cp = make_trunk([256] * 5, 0, 2)  # all streamed, 2 slots
    t.acquire(0)
    t.acquire(1)
    assert t.acquire(2, raise_on_error=False)[2] == k.K3MOE_EBUSY
    assert t.release(0) == 0
    p, r, st = t.acquire(2)
    assert ctypes.string_at(p, 1)[0] == (7 * 2 + 3) % 251
    assert t.release(3) == k.K3MOE_EINVAL  # never acquired
    t.close()


def test_failed_copy_is_reported_and_retried():
    """A failed prefetch is not an error of the request that issued it: the
    layer is copied again when it is requested, and a failure then is
    reported (and retried by the next request)."""
    cp = LogCopier(fail_on={2})  # prefix copies 0, 1; the prefetch of layer 2 fails
    t, _ = make_trunk([256] * 5, 512, 2, copier=cp)
    p, r, st = t.acquire(2)
    assert ctypes.string_at(p, 1)[0] == (7 * 2 + 3) % 251
    assert t.release(2) == 0
    # layer 3: prefetched after the acquire of 2 (copy 3), again after its
    # release (copy 4), then on demand (copy 5): all three fail
    cp = LogCopier(fail_on={3, 4, 5})
    t2, _ = make_trunk([256] * 5, 512, 2, copier=cp)
    assert t2.acquire(2)[2] == 0 and t2.release(2) == 0
    assert t2.acquire(3, raise_on_error=False)[2] == k.K3MOE_ECUDA
    p, r, st = t2.acquire(3)
    assert ctypes.string_at(p, 1)[0] == (7 * 3 + 3) % 251
    cp = LogCopier(fail_on={1})  # a prefix copy fails: no trunk
    with pytest.raises(k.K3Error):
        make_trunk([256] * 5, 512, 2, copier=cp)
    t.close()
    t2.close()


def test_refusals():
    lib = k.lib()
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(64)
    ptrs = (ctypes.c_void_p * 2)(ctypes.addressof(buf), ctypes.addressof(buf))
    cp = LogCopier()
    for sizes, pinned, ring in [((64, 60), 0, 1), ((64, 0), 0, 1), ((64, 64), 64, 0)]:
        sz = (ctypes.c_size_t * 2)(*sizes)
        assert lib.k3moe_trunk_create_with_copier(ctypes.byref(h), ptrs, sz, 2, pinned, ring,
                                                  ctypes.byref(cp.struct)) == k.K3MOE_EINVAL
    t, _ = make_trunk([256] * 3, 0, 1)
    assert t.acquire(3, raise_on_error=False)[2] == k.K3MOE_EINVAL
    assert t.acquire(-1, raise_on_error=False)[2] == k.K3MOE_EINVAL
    t.close()
