"""Pins of the oracle's SwiGLU expert, router, top-k/softmax, combine and
RMSNorm against closed forms, invariants and brute force (no GPU)."""
import math

import numpy as np
import pytest

import oracle


# ------------------------------------------------------------------ SwiGLU

def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    # sigma(ln 3) = 3/4
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    for z in [0.1, 1.0, 2.5, 7.0]:
        # silu(z) - silu(-z) = z
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14 * max(1.0, z)
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15


def _one_hot_matrix(rows, cols, cols_of_row, code, exponent=127):
    packed = np.zeros((rows, cols // 2), np.uint8)
    for r, c in enumerate(cols_of_row):
        packed[r, c // 2] |= code << (4 * (c & 1))
    scales = np.full((rows, cols // 32), exponent, np.uint8)
    return packed, scales


def test_expert_closed_form_gate_up_down_roles():
    """gate row i = 1.0 at column a_i, up row i = 2.0 at column b_i, down row r
    = 1.0 at column c_r:  y[r] = silu(x[a_{c_r}]) * 2 * x[b_{c_r}].
    A swap of gate and up, or a transposed down product, fails this."""
    d, f = 64, 32
    rng = np.random.default_rng(11)
    a = rng.integers(0, d, f)
    b = rng.integers(0, d, f)
    c = rng.integers(0, f, d)
    gp, gs = _one_hot_matrix(f, d, a, 2)   # code 2 = 1.0
    up, us = _one_hot_matrix(f, d, b, 4)   # code 4 = 2.0
    dp, ds = _one_hot_matrix(d, f, c, 2)
    ex = dict(gate_packed=gp, gate_scales=gs, up_packed=up, up_scales=us,
              down_packed=dp, down_scales=ds)
    x = rng.standard_normal(d)
    y, h = oracle.expert_forward(ex, x, want_h=True)
    for i in range(f):
        hi = x[a[i]] / (1 + math.exp(-x[a[i]])) * 2 * x[b[i]]
        assert abs(h[i] - hi) <= 1e-15 * max(1.0, abs(hi))
    for r in range(d):
        assert y[r] == h[c[r]]


def test_round_bf16_values():
    assert oracle.round_bf16(1.0) == 1.0
    assert oracle.round_bf16(1.0 + 2 ** -8) == 1.0           # tie -> even
    assert oracle.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6  # tie -> even (up)
    assert oracle.round_bf16(1.0 + 2 ** -8 + 2 ** -20) == 1.0 + 2 ** -7
    assert oracle.round_bf16(-3.0) == -3.0
    assert oracle.round_bf16(0.1) == 0.10009765625           # bf16(0.1) = 0x3DCD
    assert oracle.round_bf16(0.0) == 0.0


def test_expert_h_bf16_contract():
    """With h rounded to bf16 the one-hot expert returns bf16(h) exactly."""
    d, f = 32, 32
    idx = np.arange(f)
    gp, gs = _one_hot_matrix(f, d, idx, 2)
    up, us = _one_hot_matrix(f, d, idx, 2)
    dp, ds = _one_hot_matrix(d, f, idx, 2)
    ex = dict(gate_packed=gp, gate_scales=gs, up_packed=up, up_scales=us,
              down_packed=dp, down_scales=ds)
    x = np.linspace(-3, 3, d)
    y = oracle.expert_forward(ex, x, h_bf16=True)
    for i in range(d):
        assert y[i] == oracle.round_bf16(oracle.silu(x[i]) * x[i])


# ------------------------------------------------------------------ router

def test_bf16_values():
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC000) == -2.0
    assert oracle.bf16_value(0x3E80) == 0.25
    assert oracle.bf16_value(0x0001) == 2.0 ** -133
    assert oracle.bf16_value(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127


def test_router_orientation_one_hot():
    """logits[t][e] = sum_i W_r[e][i] x[t][i]: a one-hot x picks column i."""
    E, d = 12, 40
    rng = np.random.default_rng(5)
    Wr = rng.integers(0, 1 << 16, (E, d)).astype(np.uint16)
    Wr[(Wr & 0x7F80) == 0x7F80] = 0x3F80  # no inf/nan patterns
    x = np.zeros((2, d))
    x[0, 7] = 1.0
    x[1, 31] = -2.0
    lg = oracle.router_logits(x, Wr)
    for e in range(E):
        assert lg[0, e] == oracle.bf16_value(Wr[e, 7])
        assert lg[1, e] == -2.0 * oracle.bf16_value(Wr[e, 31])


# ------------------------------------------------------------------ top-k

def _brute_topk(scores, k):
    order = sorted(range(len(scores)), key=lambda e: (-scores[e], e))
    return sorted(order[:k])


@pytest.mark.parametrize("E,k", [(8, 3), (64, 16), (896, 16)])
def test_topk_against_full_sort(E, k):
    rng = np.random.default_rng(E)
    for trial in range(10):
        lg = rng.standard_normal(E)
        if trial % 3 == 1:
            lg = np.round(lg * 2) / 2  # many exact ties
        if trial % 3 == 2:
            lg[:] = 0.25  # all tied: the lowest ids win
        bias = rng.standard_normal(E) if trial % 2 else None
        ids, w, m = oracle.topk(lg, k, bias)
        s = lg + (bias if bias is not None else 0)
        assert list(ids[0]) == _brute_topk(list(s), k)
        chosen = set(ids[0])
        assert min(s[list(chosen)]) >= max(s[[e for e in range(E) if e not in chosen]])
        srt = sorted(s, reverse=True)
        assert m[0] == srt[k - 1] - srt[k]


def test_softmax_closed_form_and_bias_steers_selection_only():
    """Selection on logit + bias, weights from the UNBIASED logits
    ("Running Kimi K3 locally", 'How is the C engine actually built?',
    invariant 3).  logits [0, ln 3, 5], bias [10, 10, 0], k = 2: experts 0 and
    1 are chosen, weights softmax([0, ln 3]) = [1/4, 3/4]."""
    lg = np.array([0.0, math.log(3.0), 5.0])
    ids, w, m = oracle.topk(lg, 2, np.array([10.0, 10.0, 0.0]))
    assert list(ids[0]) == [0, 1]
    assert abs(w[0, 0] - 0.25) < 1e-15 and abs(w[0, 1] - 0.75) < 1e-15
    # without the bias expert 2 is chosen
    ids, w, m = oracle.topk(lg, 2)
    assert list(ids[0]) == [1, 2]
    e = math.exp(5 - math.log(3.0))
    assert abs(w[0, 1] - e / (1 + e)) < 1e-15


def test_softmax_invariants():
    rng = np.random.default_rng(9)
    lg = rng.standard_normal((20, 896)) * 3
    ids, w, _ = oracle.topk(lg, 16)
    assert np.all(np.abs(w.sum(1) - 1) < 1e-15)
    ids2, w2, _ = oracle.topk(lg + 123.0, 16)  # shift invariance
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-12, atol=0)
    # weights follow the logits' order
    for t in range(20):
        order = np.argsort(lg[t, ids[t]])
        assert np.all(np.diff(w[t, order]) >= 0)


# --------------------------------------------------------- sigmoid router

def _logistic(z):
    """The logistic function through tanh, an identity independent of the
    oracle's 1 / (1 + e^-z): sigma(z) = (1 + tanh(z / 2)) / 2."""
    return 0.5 * (1.0 + np.tanh(np.asarray(z, np.float64) / 2.0))


def test_sigmoid_router_selects_on_sigmoid_plus_bias():
    """Selection on sigmoid(logit) + bias, weights the unbiased sigmoid
    scores ("Running Kimi K3 locally", 'How is the C engine actually built?',
    invariant 3).  logits [3, 0, -1], bias [0, 0.6, 0], k = 1: sigmoid(3) =
    0.9526 < sigmoid(0) + 0.6 = 1.1, so expert 1 is chosen, with weight
    sigmoid(0) = 1/2 (not the biased 1.1).  Selection on logit + bias, or on
    sigmoid(logit + bias), would choose expert 0."""
    lg = np.array([3.0, 0.0, -1.0])
    b = np.array([0.0, 0.6, 0.0])
    for router in ("sigmoid", "sigmoid_norm"):
        ids, w, m = oracle.topk(lg, 1, b, router)
        assert list(ids[0]) == [1]
        assert w[0, 0] == (0.5 if router == "sigmoid" else 1.0)
        assert abs(m[0] - (1.1 - _logistic(3.0))) < 1e-15
    assert list(oracle.topk(lg, 1, b)[0][0]) == [0]  # the softmax router's choice
    # k = 2: experts 0 and 1, weights sigmoid(3) and 1/2
    ids, w, _ = oracle.topk(lg, 2, b, "sigmoid")
    assert list(ids[0]) == [0, 1]
    assert abs(w[0, 0] - _logistic(3.0)) < 1e-15 and w[0, 1] == 0.5


@pytest.mark.parametrize("E,k", [(8, 3), (64, 16), (896, 16)])
def test_sigmoid_router_against_full_sort(E, k):
    rng = np.random.default_rng(100 + E)
    for trial in range(10):
        lg = rng.standard_normal(E) * 2
        if trial % 3 == 1:
            lg = np.round(lg * 2) / 2  # many exact ties
        bias = rng.standard_normal(E) * 0.1 if trial % 2 else None
        ids, w, m = oracle.topk(lg, k, bias, "sigmoid")
        s = _logistic(lg) + (bias if bias is not None else 0)
        if trial % 3 != 1:  # no near-ties: the tanh form orders exactly alike
            assert list(ids[0]) == _brute_topk(list(s), k)
            srt = sorted(s, reverse=True)
            assert abs(m[0] - (srt[k - 1] - srt[k])) < 1e-14
        # weights: the unbiased scores of the chosen experts
        assert np.allclose(w[0], _logistic(lg[ids[0]]), rtol=1e-14, atol=0)
        _, wn, _ = oracle.topk(lg, k, bias, "sigmoid_norm")
        assert abs(wn[0].sum() - 1.0) < 1e-15
        assert np.allclose(wn[0], w[0] / w[0].sum(), rtol=1e-14, atol=0)


def test_sigmoid_router_without_bias_selects_like_the_softmax_router():
    """The logistic function is increasing: with no bias the chosen set is
    that of the (pinned) softmax router, ties included."""
    rng = np.random.default_rng(31)
    lg = rng.standard_normal((40, 896)) * 1.7
    lg[::5] = np.round(lg[::5] * 4) / 4
    assert np.array_equal(oracle.topk(lg, 16, None, "sigmoid")[0], oracle.topk(lg, 16)[0])


def test_sigmoid_router_bias_steers_selection_only():
    """Two biases that choose the same experts give the same weights; the
    weights never depend on the bias.  A router that took its weights from
    the biased scores fails these checks (planted below)."""
    rng = np.random.default_rng(32)
    lg = rng.standard_normal((30, 896)) * 1.7
    b1 = rng.standard_normal(896) * 0.05
    ids1, w1, _ = oracle.topk(lg, 16, b1, "sigmoid")
    ids2, w2, _ = oracle.topk(lg, 16, b1 + 0.37, "sigmoid")  # a constant shift keeps the choice
    assert np.array_equal(ids1, ids2) and np.array_equal(w1, w2)
    for t in range(30):
        assert np.allclose(w1[t], _logistic(lg[t, ids1[t]]), rtol=1e-14, atol=0)
    collapsed = w1 + b1[ids1]  # weights from the biased score: the mistake
    assert not np.allclose(collapsed, _logistic(np.take_along_axis(lg, ids1.astype(np.int64), 1)),
                           rtol=1e-6, atol=0)


# ------------------------------------------------------------------ layer

def _rand_expert(rng, d, f):
    return dict(gate_packed=rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
                gate_scales=rng.integers(120, 131, (f, d // 32), dtype=np.uint8),
                up_packed=rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
                up_scales=rng.integers(120, 131, (f, d // 32), dtype=np.uint8),
                down_packed=rng.integers(0, 256, (d, f // 2), dtype=np.uint8),
                down_scales=rng.integers(120, 131, (d, f // 32), dtype=np.uint8))


def test_layer_identical_experts_reduce_to_one_expert():
    """If every expert is the same, the softmax weights sum to 1 and the layer
    output equals that one expert's output."""
    rng = np.random.default_rng(2)
    d, f, E, k = 64, 32, 10, 4
    ex = _rand_expert(rng, d, f)
    Wr = (rng.standard_normal((E, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = rng.standard_normal((3, d))
    out, ids, w, _ = oracle.layer_forward(x, Wr, k, {e: ex for e in range(E)})
    for t in range(3):
        y = oracle.expert_forward(ex, x[t])
        assert np.allclose(out[t], y, rtol=1e-13, atol=1e-12 * np.abs(y).max())


def test_layer_is_weighted_sum_of_selected_experts():
    """Linearity of the combine: scaling one expert's down matrix by 2 (its
    exponents + 1) adds exactly w_j * y_j to the output."""
    rng = np.random.default_rng(4)
    d, f, E, k = 64, 32, 6, 3
    exs = {e: _rand_expert(rng, d, f) for e in range(E)}
    Wr = (rng.standard_normal((E, d)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = rng.standard_normal((1, d))
    out, ids, w, _ = oracle.layer_forward(x, Wr, k, exs)
    j = 1
    e = int(ids[0, j])
    ex2 = dict(exs[e])
    ex2["down_scales"] = exs[e]["down_scales"] + 1
    exs2 = dict(exs)
    exs2[e] = ex2
    out2, ids2, w2, _ = oracle.layer_forward(x, Wr, k, exs2)
    assert np.array_equal(ids, ids2)
    y = oracle.expert_forward(exs[e], x[0])
    assert np.allclose(out2[0] - out[0], w[0, j] * y, rtol=1e-9, atol=1e-9 * np.abs(y).max())


@pytest.mark.parametrize("h_bf16", [False, True])
def test_grouped_combine_equals_per_pair_combine(h_bf16):
    """The grouped form (each expert dequantised once, all its tokens in one
    fp64 matrix product) reaches the per-pair combine's result up to the
    order of fp64 sums; a planted mistake (one pair's weight dropped) is
    seen."""
    rng = np.random.default_rng(11)
    d, f, E, k, T = 96, 64, 7, 3, 9
    exs = {e: _rand_expert(rng, d, f) for e in range(E)}
    x = rng.standard_normal((T, d))
    ids = np.stack([np.sort(rng.choice(E, k, replace=False)) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k))
    ref = oracle.combine(x, ids, w, exs, E, h_bf16)
    got = oracle.combine_grouped(x, ids, w, lambda e: exs[e], h_bf16)
    scale = np.abs(ref).max()
    assert np.max(np.abs(got - ref)) <= 1e-12 * scale
    w2 = w.copy()
    w2[4, 1] = 0.0
    bad = oracle.combine_grouped(x, ids, w2, lambda e: exs[e], h_bf16)
    assert np.max(np.abs(bad - ref)) > 1e-3 * scale


# ----------------------------------------------------------------- rmsnorm

def test_rmsnorm_closed_forms_eps_inside_sqrt():
    eps = 1e-6
    y = oracle.rmsnorm(np.array([3.0, 4.0]), eps)
    assert np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5 + eps), rtol=1e-15)
    # a single element equal to sqrt(eps): y = 1/sqrt(2) only if eps is
    # inside the square root (176 KB Engine, 'What byte-identical actually
    # costs'); outside it would give ~1.
    y = oracle.rmsnorm(np.array([math.sqrt(eps)]), eps)
    assert abs(y[0] - 1 / math.sqrt(2)) < 1e-12
    y = oracle.rmsnorm(np.zeros(5), eps)
    assert not y.any()
    x = np.random.default_rng(1).standard_normal(7168)
    y = oracle.rmsnorm(x, 0.0)
    assert abs(np.mean(y ** 2) - 1) < 1e-12
