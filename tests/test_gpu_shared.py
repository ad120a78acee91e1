"""GPU parity of the bf16 shared (always-on) experts (k3moe_shared_forward)
against the oracle's fp64 definition, alone and inside the streamed decode,
where each layer's shared experts come from its dense-trunk bytes through
the trunk streamer (a resident prefix plus ring slots)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import TOL, rel_err, router_tensor
from mxfp4_routed_expert_select_gb300 import k3moe as k
from test_gpu_stream import EPS, POOL, HostLayers

pytestmark = pytest.mark.gpu


def _blob(ex):
    """Device blob gate | up | down of one shared expert."""
    raw = np.concatenate([ex["gate"].ravel(), ex["up"].ravel(), ex["down"].ravel()]).view(np.uint8)
    return torch.from_numpy(raw.copy()).cuda()


def _case(n, d, f, T, pool, accumulate):
    exs = [synth.shared_expert(pool, 0, s, d, f) for s in range(n)]
    blobs = [_blob(e) for e in exs]
    views = [k.shared_expert_view(b.data_ptr(), d, f) for b in blobs]
    X = synth.tokens_f32(pool, T, d)
    Xd = torch.from_numpy(X).cuda()
    base = synth.tokens_f32(pool, T, d, t0=1000)
    out = torch.from_numpy(base.copy()).cuda()
    ws = torch.empty(k.shared_workspace(n, f) // 4, dtype=torch.float32, device="cuda")
    k.shared_forward(out, Xd, T, views, d, f, ws, accumulate=accumulate)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref = oracle.shared_forward(X.astype(np.float64), exs)
    if accumulate:
        ref = ref + base
    for t in range(T):
        e = rel_err(got[t], ref[t])
        assert e <= TOL, (t, e)
    return max(rel_err(got[t], ref[t]) for t in range(T))


@pytest.mark.parametrize("n,d,f,T,acc", [(1, 512, 256, 1, False), (3, 512, 256, 4, True),
                                         (4, 1024, 512, 9, False), (2, 768, 512, 2, True)])
def test_shared_forward_small(n, d, f, T, acc):
    _case(n, d, f, T, 51, acc)


@pytest.mark.parametrize("T", [1, 5])
def test_shared_forward_full_shape_two_experts(T):
    """d = 7168, f = 1536, the pages' two shared experts; T = 5 spans two
    launch groups of tokens."""
    err = _case(2, 7168, 1536, T, 52, accumulate=(T == 5))
    print("shared experts d=7168 f=1536 T=%d: max rel err %.2e" % (T, err))


def test_shared_forward_refuses_bad_calls():
    d, f = 512, 256
    ex = synth.shared_expert(53, 0, 0, d, f)
    b = _blob(ex)
    v = k.shared_expert_view(b.data_ptr(), d, f)
    x = torch.zeros((1, d), dtype=torch.float32, device="cuda")
    out = torch.zeros_like(x)
    ws = torch.empty(k.shared_workspace(4, f) // 4 + 16, dtype=torch.float32, device="cuda")
    for views, dd, ff in (([v] * 5, d, f), ([v], 500, f), ([v], d, 250)):
        with pytest.raises(k.K3Error) as ei:
            k.shared_forward(out, x, 1, views, dd, ff, ws)
        assert ei.value.status == k.K3MOE_EINVAL
    assert k.shared_expert_bytes(7168, 1536) == 6 * 7168 * 1536


class SharedLayers(HostLayers):
    """HostLayers plus two bf16 shared experts per layer, one pinned host
    buffer per layer (the trunk's bytes)."""

    def __init__(self, n_layers, E, K, d, f, n_shared=2):
        super().__init__(n_layers, E, K, d, f)
        self.ns = n_shared
        self.shared = [[synth.shared_expert(POOL, l, s, d, f) for s in range(n_shared)] for l in range(n_layers)]
        self.trunk_host = []
        for l in range(n_layers):
            raw = np.concatenate([np.concatenate([e["gate"].ravel(), e["up"].ravel(), e["down"].ravel()])
                                  for e in self.shared[l]]).view(np.uint8)
            t = torch.from_numpy(raw.copy()).pin_memory()
            self.trunk_host.append(t)

    def chain(self, x):
        x = np.asarray(x, np.float64).copy()
        ids_all, margins = [], []
        for l in range(self.nl):
            u = oracle.rmsnorm(x, EPS)
            lg = oracle.router_logits(u, self.Wr[l])
            ids, w, m = oracle.topk(lg, self.K, self.bias[l])
            ex = {int(e): self.planes(l, int(e)) for e in ids[0]}
            x = x + oracle.combine(u[None], ids, w, ex, self.E)[0] + oracle.shared_forward(u[None], self.shared[l])[0]
            ids_all.append(ids[0])
            margins.append(m[0])
        return x, np.stack(ids_all), np.array(margins)


def test_stream_decode_with_shared_experts_from_the_trunk():
    """3 layers, 40 experts each (top-4), two shared experts per layer read
    from the trunk: one layer resident, two streamed through two ring slots."""
    hl = SharedLayers(3, 40, 4, 1024, 512)
    T = 4
    X, refs, rids = [], [], []
    for t in range(T):
        for s in range(40):
            x = synth.token_f32(POOL, t, hl.d, s)
            o, i, m = hl.chain(x)
            if np.all(m >= 1e-3):
                break
        X.append(x)
        refs.append(o)
        rids.append(i)
    X = np.stack(X)
    lb = [t.numel() for t in hl.trunk_host]
    trunk = k.Trunk([t.data_ptr() for t in hl.trunk_host], lb, lb[0], 2)
    cache = k.Cache(30 * hl.eb, hl.eb, hl.ptrs(), hl.nl, hl.E)
    layers = hl.device_layers()
    Xd = torch.from_numpy(X).cuda()
    out = torch.empty_like(Xd)
    ids, hits = k.stream_decode(layers, cache, Xd, T, out, EPS, trunk=trunk, n_shared=hl.ns)
    torch.cuda.synchronize()
    assert np.array_equal(ids, np.stack(rids))
    got = out.cpu().numpy()
    for t in range(T):
        e = rel_err(got[t], refs[t])
        assert e <= TOL, (t, e)
    st = trunk.stats()
    assert st["requests"] == T * hl.nl and st["pinned_layers"] == 1
    assert k.device_error() == 0
    for L in layers:
        L.close()
    cache.close()
    trunk.close()
