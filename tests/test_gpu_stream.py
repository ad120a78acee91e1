"""GPU parity of the host-streamed decode loop (k3moe_stream_decode): several
MoE layers whose experts live in pinned host memory behind the HBM LRU cache,
RMSNorm + residual between layers.  Expected values come from the oracle's
chain (rmsnorm -> router -> top-k -> combine -> residual, fp64) and from its
LRU replay of the same key sequence."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import TOL, rel_err, router_tensor
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu

EPS = 1e-6
POOL = 21


class HostLayers:
    """n_layers x E experts as blobs in one pinned host tensor, plus each
    layer's router and Zipf selection bias."""

    def __init__(self, n_layers, E, K, d, f, zipf=True):
        self.nl, self.E, self.K, self.d, self.f = n_layers, E, K, d, f
        self.eb = k.expert_bytes(d, f)
        self.host = torch.empty((n_layers * E, self.eb), dtype=torch.uint8).pin_memory()
        stage = torch.empty((self.eb,), dtype=torch.uint8, device="cuda")
        for l in range(n_layers):
            for e in range(E):
                k.pack_expert(stage, synth.expert(POOL, l, e, d, f), d, f)
                torch.cuda.synchronize()
                self.host[l * E + e].copy_(stage.cpu())
        self.Wr = [synth.router_bf16(POOL, l, E, d) for l in range(n_layers)]
        self.bias = [synth.bias_zipf(POOL, l, E) if zipf else None for l in range(n_layers)]
        self._planes = {}

    def planes(self, l, e):
        key = (l, e)
        if key not in self._planes:
            if len(self._planes) > 96:
                self._planes.clear()
            self._planes[key] = synth.expert(POOL, l, e, self.d, self.f)
        return self._planes[key]

    def ptrs(self):
        base = self.host.data_ptr()
        return [base + q * self.eb for q in range(self.nl * self.E)]

    def device_layers(self):
        out = []
        for l in range(self.nl):
            b = None if self.bias[l] is None else torch.from_numpy(
                np.ascontiguousarray(self.bias[l], np.float32)).cuda()
            out.append(k.Layer(self.E, self.K, self.d, self.f, router_tensor(self.Wr[l]), None, b,
                               max_tokens=1))
        return out

    def chain(self, x):
        """Oracle: the token through every layer; (out, ids [L,K], margins [L])."""
        x = np.asarray(x, np.float64).copy()
        ids_all, margins = [], []
        for l in range(self.nl):
            u = oracle.rmsnorm(x, EPS)
            lg = oracle.router_logits(u, self.Wr[l])
            ids, w, m = oracle.topk(lg, self.K, self.bias[l])
            ex = {int(e): self.planes(l, int(e)) for e in ids[0]}
            x = x + oracle.combine(u[None], ids, w, ex, self.E)[0]
            ids_all.append(ids[0])
            margins.append(m[0])
        return x, np.stack(ids_all), np.array(margins)


def margin_tokens(hl, T, gap=1e-3, max_tries=40):
    """Tokens whose every layer's rank-K / rank-K+1 gap is at least `gap`
    (a token is redrawn from its next substream otherwise)."""
    X, outs, ids = [], [], []
    for t in range(T):
        for s in range(max_tries):
            x = synth.token_f32(POOL, t, hl.d, s)
            o, i, m = hl.chain(x)
            if np.all(m >= gap):
                break
        else:
            raise RuntimeError("no margin token")
        X.append(x)
        outs.append(o)
        ids.append(i)
    return np.stack(X), np.stack(outs), np.stack(ids)


def run(hl, cache, X):
    T = X.shape[0]
    layers = hl.device_layers()
    Xd = torch.from_numpy(X).cuda()
    out = torch.empty_like(Xd)
    ids, hits = k.stream_decode(layers, cache, Xd, T, out, EPS)
    torch.cuda.synchronize()
    for L in layers:
        L.close()
    return out.cpu().numpy(), ids, hits


@pytest.fixture(scope="module")
def small():
    hl = HostLayers(3, 40, 4, 1024, 512)
    X, ref, rids = margin_tokens(hl, 8)
    return hl, X, ref, rids


@pytest.mark.parametrize("slots", [12, 30, 120])
def test_stream_small_matches_oracle_chain_and_lru(small, slots):
    hl, X, ref, rids = small
    cache = k.Cache(slots * hl.eb, hl.eb, hl.ptrs(), hl.nl, hl.E)
    out, ids, hits = run(hl, cache, X)
    T = X.shape[0]
    assert np.array_equal(ids, rids)
    for t in range(T):
        e = rel_err(out[t], ref[t])
        assert e <= TOL, (t, e)
    keys = (np.arange(hl.nl)[None, :, None] * hl.E + rids).reshape(-1).astype(np.int64)
    nh, rhit = oracle.cache_lru(keys, np.full(T * hl.nl, hl.K, np.int32), slots)
    assert np.array_equal(hits.reshape(-1), rhit)
    st = cache.stats()
    assert st["lookups"] == keys.size and st["hits"] == nh
    assert st["h2d_bytes"] == (keys.size - nh) * hl.eb
    if slots >= hl.nl * hl.E:
        assert st["evictions"] == 0
    cache.close()


def test_stream_refuses_a_cache_too_small_for_one_batch(small):
    hl, X, _, _ = small
    cache = k.Cache(3 * hl.eb, hl.eb, hl.ptrs(), hl.nl, hl.E)  # 3 slots < top-4
    layers = hl.device_layers()
    Xd = torch.from_numpy(X[:1]).cuda()
    out = torch.empty_like(Xd)
    with pytest.raises(k.K3Error) as ei:
        k.stream_decode(layers, cache, Xd, 1, out, EPS)
    assert ei.value.status == k.K3MOE_EBUSY
    for L in layers:
        L.close()
    cache.close()


def test_stream_full_shape_two_layers():
    """d=7168, f=1536, top-16 of 64 experts per layer, a cache of 40 slots
    (less than one layer's experts) so that tokens evict each other."""
    hl = HostLayers(2, 64, 16, 7168, 1536)
    X, ref, rids = margin_tokens(hl, 3)
    cache = k.Cache(40 * hl.eb, hl.eb, hl.ptrs(), hl.nl, hl.E)
    out, ids, hits = run(hl, cache, X)
    assert np.array_equal(ids, rids)
    for t in range(X.shape[0]):
        e = rel_err(out[t], ref[t])
        assert e <= TOL, (t, e)
    keys = (np.arange(hl.nl)[None, :, None] * hl.E + rids).reshape(-1).astype(np.int64)
    nh, rhit = oracle.cache_lru(keys, np.full(X.shape[0] * hl.nl, hl.K, np.int32), 40)
    assert np.array_equal(hits.reshape(-1), rhit)
    cache.close()
