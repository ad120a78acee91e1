"""The batch-1 layer's selection over many router shapes and tie patterns,
against the oracle's top-k: ids bit-exact, combine weights close.

Router rows are power-of-two multiples c_r v of one row v, c_r from
{-4, -2, -1, 0, 1, 2, 4} in a fixed pattern, so every fp32 logit is exactly
c_r times one dot product (power-of-two scaling commutes with rounding) and
rows with equal c_r tie exactly on both sides.  "cont" uses independent rows
(no ties), "groups" the multiples, "equal" one row for every expert (every
logit ties: the selection's many-ties fallback).  The cases cover E from 8
to 1024, k from 1 to 16, a selection bias of small integers and the sigmoid
rule.  A case whose k-th and (k+1)-th selection keys differ by less than
1e-4 in fp64 without being equal takes the next token, so that fp32
rounding cannot move the boundary.  Only
the selection is checked: the experts are a small pool reused under many
ids."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import Pool, router_tensor
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu

D, F, NPOOL = 512, 512, 16
MULT = np.array([-4.0, -2.0, -1.0, 0.0, 1.0, 2.0, 4.0])


@pytest.fixture(scope="module")
def pool():
    return Pool(21, 0, NPOOL, D, F)


def _router(E, pattern):
    if pattern == "cont":
        return synth.router_bf16(21, 1, E, D)
    v = synth.router_bf16(21, 2, 1, D)[0]
    vf = (v.astype(np.uint32) << 16).view(np.float32)
    c = np.ones(E) if pattern == "equal" else MULT[(np.arange(E) * 5 + E) % len(MULT)]
    rows = (c[:, None] * vf[None, :]).astype(np.float32)  # exact: power-of-two multiples of bf16 values
    bits = rows.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0)
    return (bits >> 16).astype(np.uint16)


def _keys(lg, bias, rule):
    s = lg if rule == "softmax" else 1.0 / (1.0 + np.exp(-lg))
    return s if bias is None else s + bias


def _boundary_ok(keys, K):
    """The k-th and (k+1)-th largest keys either tie exactly (equal rows and
    equal bias: the same computation on both sides) or are 1e-4 apart."""
    if K >= keys.size:
        return True
    s = np.sort(np.round(keys, 12))[::-1]
    return s[K - 1] == s[K] or s[K - 1] - s[K] > 1e-4


CASES = [
    # E, k, pattern, bias, rule
    (8, 1, "cont", False, "softmax"),
    (8, 8, "groups", False, "softmax"),
    (33, 4, "groups", True, "softmax"),
    (33, 16, "equal", False, "softmax"),
    (64, 8, "cont", True, "sigmoid"),
    (130, 16, "groups", False, "softmax"),
    (130, 5, "equal", True, "softmax"),
    (257, 16, "cont", False, "softmax"),
    (257, 3, "groups", True, "sigmoid"),
    (512, 16, "groups", False, "sigmoid"),
    (512, 8, "equal", False, "softmax"),
    (896, 16, "cont", False, "softmax"),
    (896, 16, "groups", False, "softmax"),
    (896, 16, "groups", True, "softmax"),
    (896, 16, "equal", True, "sigmoid"),
    (896, 1, "groups", False, "softmax"),
    (1024, 16, "cont", True, "softmax"),
    (1024, 12, "groups", False, "softmax"),
    (1024, 16, "equal", False, "softmax"),
]


@pytest.mark.parametrize("E,K,pattern,use_bias,rule", CASES)
def test_selection_cases(pool, E, K, pattern, use_bias, rule):
    Wr_bits = _router(E, pattern)
    bias = ((np.arange(E) * 7) % 3).astype(np.float32) if use_bias else None
    views = [pool.views[e % NPOOL] for e in range(E)]
    L = k.Layer(E, K, D, F, router_tensor(Wr_bits), views,
                None if bias is None else torch.from_numpy(bias).cuda(), max_tokens=1)
    if rule == "sigmoid":
        L.set_option(k.K3MOE_OPT_SIGMOID_ROUTER, 1)
    assert L.mx_t1()
    b64 = None if bias is None else bias.astype(np.float64)
    for t in range(20):
        x = synth.token_f32(21, t, D, sub=E)
        lg = oracle.router_logits(x[None], Wr_bits)
        if _boundary_ok(_keys(lg[0], b64, rule), K):
            break
    else:
        pytest.fail("no token with a clear selection boundary")
    rids, rw, _ = oracle.topk(lg, K, b64, router=rule)
    out = torch.empty((1, D), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, K), dtype=torch.int32, device="cuda")
    w = torch.empty((1, K), dtype=torch.float32, device="cuda")
    L.forward(torch.from_numpy(x[None]).cuda(), 1, out, ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), rids), (ids.cpu().numpy(), rids)
    assert np.allclose(w.cpu().numpy(), rw, rtol=2e-4, atol=1e-7)
    assert k.device_error() == 0
    L.close()
