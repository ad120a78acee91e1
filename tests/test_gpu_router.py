"""GPU parity of the sigmoid router variant (K3MOE_OPT_SIGMOID_ROUTER):
selection on sigmoid(logit) + bias, combine weights the unbiased sigmoid
scores, as they are or renormalised ("Running Kimi K3 locally", "How is the
C engine actually built?", invariant 3), on every forward path, against the
fp64 oracle: ids bit-exact on margin-checked tokens, weights and outputs
within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import TOL, Pool, margin_subs, rel_err, router_tensor, tokens, tokens_device
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu

PATHS = [("mx", 1, False), ("fused", 1, False), ("unfused", 1, False), ("unfused", 1, True),
         ("multi", 5, False), ("multi", 130, True)]


@pytest.fixture(scope="module")
def pool():
    E, d, f = 48, 1024, 512
    return Pool(6, 0, E, d, f), synth.router_bf16(6, 0, E, d), synth.bias_normal(6, 0, E)


def _layer(pool, Wr, bias, K, T, path, router):
    p = pool
    L = k.Layer(p.E, K, p.d, p.f, Wr, p.views, bias, max_tokens=T)
    L.set_option(k.K3MOE_OPT_SIGMOID_ROUTER, 1)
    L.set_option(k.K3MOE_OPT_SIGMOID_NORM, 1 if router == "sigmoid_norm" else 0)
    L.set_option(k.K3MOE_OPT_MX, 1 if path == "mx" else 0)
    L.set_option(k.K3MOE_OPT_FUSED_T1, 1 if path == "fused" else 0)
    if T == 1:
        assert L.mx_t1() == (path == "mx") and L.fused_t1() == (path == "fused")
    return L


def _run(L, X, T, K):
    out = torch.empty((T, L.d), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    L.forward(X, T, out, ids, w)
    torch.cuda.synchronize()
    assert k.device_error() == 0
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("router", ["sigmoid", "sigmoid_norm"])
@pytest.mark.parametrize("path,T,bf16", PATHS)
def test_sigmoid_router_matches_oracle(pool, path, T, bf16, router):
    p, Wr_bits, bias = pool
    K = 8
    b = (0.05 * bias).astype(np.float32)  # scores lie in (0, 1): a bias of their spread
    subs = margin_subs(6, T, p.d, Wr_bits, K, b, bf16=bf16, router=router)
    Xd = tokens(6, np.arange(T), p.d, subs, bf16)
    X = tokens_device(6, T, p.d, subs, bf16)
    L = _layer(p, router_tensor(Wr_bits), torch.from_numpy(b).cuda(), K, T, path, router)
    out, ids, w = _run(L, X, T, K)
    lg = oracle.router_logits(Xd, Wr_bits)
    rids, rw, m = oracle.topk(lg, K, b.astype(np.float64), router)
    assert np.all(m >= 1e-3)
    assert np.array_equal(ids, rids)
    assert np.allclose(w, rw, rtol=2e-4, atol=1e-7)
    for t in (range(T) if T <= 5 else (0, 63, T - 1)):
        ref = oracle.combine(Xd[t:t + 1], rids[t:t + 1], rw[t:t + 1], p.experts(rids[t]), p.E)[0]
        assert rel_err(out[t], ref) <= TOL, t
    L.close()


@pytest.mark.parametrize("router", ["sigmoid", "sigmoid_norm"])
@pytest.mark.parametrize("path,T", [("mx", 1), ("fused", 1), ("unfused", 1), ("multi", 3)])
def test_bias_selects_and_the_unbiased_scores_weigh(pool, path, T, router):
    """W_r = 0: every logit is 0 and every score sigmoid(0) = 1/2.  A bias
    that favours the top ids chooses them; their weights stay 1/2 (or 1/K
    renormalised), never the biased scores."""
    p, _, _ = pool
    K = 8
    zero = torch.zeros((p.E, p.d), dtype=torch.int16, device="cuda")
    bb = torch.from_numpy(np.arange(p.E, dtype=np.float32) * 0.01).cuda()
    L = _layer(p, zero, bb, K, T, path, router)
    X = tokens_device(6, T, p.d, list(range(T)))
    out, ids, w = _run(L, X, T, K)
    assert np.array_equal(ids, np.tile(np.arange(p.E - K, p.E), (T, 1)))
    assert np.allclose(w, 0.5 if router == "sigmoid" else 1.0 / K, rtol=1e-6, atol=0)
    L.close()
