"""Pins of the oracle's MXFP4 quantisation of activations (the OCP
Microscaling v1.0 conversion, a reading: the pages quantise only weights) and
of the expert forward that uses it, against an independent brute-force
quantiser, closed forms and special cases (no GPU)."""
import math

import numpy as np
import pytest

import oracle

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _brute_block(x):
    """Scale from log2 of the block maximum; each value to the nearest grid
    magnitude by exhaustive search, ties to the even code."""
    x = np.asarray(x, np.float32).astype(np.float64)
    if not np.all(np.isfinite(x)):
        return 255, None
    amax = np.max(np.abs(x))
    e = 0 if amax == 0 else int(min(max(math.floor(np.log2(amax)) - 2 + 127, 0), 254))
    out = []
    for v in np.abs(x) * 2.0 ** (127 - e):
        dist = np.abs(GRID - v)
        best = [c for c in range(8) if dist[c] == dist.min()]
        c = min(best, key=lambda c: (c % 2, c))  # the even code of a tie
        out.append(c)
    codes = np.array(out, np.uint8) | (np.signbit(x).astype(np.uint8) << 3)
    return e, codes


def _blocks(rng, n):
    """Blocks over many magnitudes, with exact midpoints planted."""
    out = []
    for i in range(n):
        k = int(rng.integers(-40, 40))
        b = rng.standard_normal(32) * 2.0 ** k
        if i % 3 == 0:  # plant midpoints of the block's grid
            s = 2.0 ** (math.floor(math.log2(np.max(np.abs(b)))) - 2)
            mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]) * s
            b[1:8] = mids * np.where(rng.integers(0, 2, 7) == 1, 1, -1)
        out.append(b.astype(np.float32))
    return out


def test_quantisation_against_brute_force():
    rng = np.random.default_rng(41)
    for b in _blocks(rng, 300):
        xq, codes, sc = oracle.mx_quantize(b)
        e, want = _brute_block(b)
        assert sc[0] == e
        assert np.array_equal(codes, want)
        assert np.array_equal(xq, [oracle.e2m1_value(c) * 2.0 ** (e - 127) for c in codes])


def test_ties_go_to_the_even_code_and_large_values_saturate():
    # block maximum 4: scale 2^0, so the block's values are on the grid's own scale
    x = np.zeros(32, np.float32)
    x[:8] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.0]
    xq, codes, sc = oracle.mx_quantize(x)
    assert sc[0] == 127
    assert list(xq[:8]) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 4.0]
    # maximum 7 * 2^-3: floor(log2) = -1, scale 2^-3, 7 saturates to 6
    x = np.zeros(32, np.float32)
    x[0], x[1] = 7 * 0.125, -7 * 0.125
    xq, codes, sc = oracle.mx_quantize(x)
    assert sc[0] == 124 and xq[0] == 0.75 and xq[1] == -0.75
    assert codes[0] == 7 and codes[1] == 15


def test_grid_values_are_kept_exactly():
    """A block whose largest magnitude is 4 or 6 times 2^s has scale 2^s, so
    every value on that block's grid is reproduced."""
    rng = np.random.default_rng(42)
    for s in (-126, -60, -3, 0, 5, 90, 125):
        c = rng.integers(0, 16, 32)
        c[int(rng.integers(0, 32))] = 7 if s % 2 else 6
        x = np.array([oracle.e2m1_value(v) * 2.0 ** s for v in c], np.float32)
        xq, codes, sc = oracle.mx_quantize(x)
        assert sc[0] == s + 127
        assert np.array_equal(xq, x.astype(np.float64))
        assert np.array_equal(oracle.mx_quantize(xq.astype(np.float32))[0], xq)  # idempotent


def test_special_blocks():
    z = np.zeros(32, np.float32)
    xq, codes, sc = oracle.mx_quantize(z)
    assert sc[0] == 0 and not xq.any() and not codes.any()
    neg = -np.full(32, 1e-3, np.float32)
    neg[0] = -1.0  # -1e-3 rounds to -0: code 8
    xq, codes, sc = oracle.mx_quantize(neg)
    assert codes[1] == 8 and xq[1] == 0.0
    for bad in (np.nan, np.inf, -np.inf):
        b = np.ones(32, np.float32)
        b[5] = bad
        xq, codes, sc = oracle.mx_quantize(b)
        assert sc[0] == 255 and np.all(np.isnan(xq))
    # tiny: the exponent clamps at 0 (scale 2^-127); huge: at 254 (2^127)
    tiny = np.full(32, 2.0 ** -140, np.float32)
    xq, _, sc = oracle.mx_quantize(tiny)
    assert sc[0] == 0 and not xq.any()  # 2^-140 / 2^-127 = 2^-13 rounds to 0
    huge = np.full(32, 3e38, np.float32)
    xq, _, sc = oracle.mx_quantize(huge)
    assert sc[0] == 252 and np.all(xq == 6.0 * 2.0 ** 125)


def test_error_bound():
    """|x - q(x)| <= 2^s where the scaled value is within the grid (half the
    largest gap, 4 to 6), and <= 2 * 2^s where it saturates (up to 8)."""
    rng = np.random.default_rng(43)
    for b in _blocks(rng, 200):
        xq, _, sc = oracle.mx_quantize(b)
        s = 2.0 ** (int(sc[0]) - 127)
        err = np.abs(b.astype(np.float64) - xq)
        inside = np.abs(b.astype(np.float64)) <= 6 * s
        assert np.all(err[inside] <= s) and np.all(err <= 2 * s)


@pytest.mark.parametrize("d,f", [(64, 32), (256, 128)])
def test_expert_forward_mxq_is_the_composition(d, f):
    """y = W_down q(fp32(silu(W_gate q(x)) * (W_up q(x)))), built here from
    the separately pinned pieces (quantiser, packed matvec, SiLU)."""
    rng = np.random.default_rng(d)
    ex = dict(gate_packed=rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
              gate_scales=rng.integers(120, 131, (f, d // 32), dtype=np.uint8),
              up_packed=rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
              up_scales=rng.integers(120, 131, (f, d // 32), dtype=np.uint8),
              down_packed=rng.integers(0, 256, (d, f // 2), dtype=np.uint8),
              down_scales=rng.integers(120, 131, (d, f // 32), dtype=np.uint8))
    x = rng.standard_normal(d).astype(np.float32)
    xq = oracle.mx_quantize(x)[0]
    g = oracle.matvec(ex["gate_packed"], ex["gate_scales"], xq)
    u = oracle.matvec(ex["up_packed"], ex["up_scales"], xq)
    h = np.array([oracle.silu(a) * b for a, b in zip(g, u)], np.float32)
    want = oracle.matvec(ex["down_packed"], ex["down_scales"], oracle.mx_quantize(h)[0])
    got = oracle.expert_forward_mxq(ex, x)
    assert np.allclose(got, want, rtol=1e-13, atol=0)
    # and it differs from the exact forward by the quantisation error only
    exact = oracle.expert_forward(ex, x.astype(np.float64))
    rel = np.max(np.abs(got - exact)) / np.max(np.abs(exact))
    assert 1e-4 < rel < 0.5


def test_grouped_mxq_combine_equals_the_per_pair_forward():
    """The grouped form (each expert's tokens in one fp64 matrix product) is
    the weighted sum of expert_forward_mxq over the chosen experts, up to the
    order of fp64 sums; a planted mistake (a pair's weight dropped) is seen."""
    rng = np.random.default_rng(21)
    d, f, E, k, T = 128, 64, 6, 3, 7
    exs = {}
    for e in range(E):
        exs[e] = dict(gate_packed=rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
                      gate_scales=rng.integers(120, 131, (f, d // 32), dtype=np.uint8),
                      up_packed=rng.integers(0, 256, (f, d // 2), dtype=np.uint8),
                      up_scales=rng.integers(120, 131, (f, d // 32), dtype=np.uint8),
                      down_packed=rng.integers(0, 256, (d, f // 2), dtype=np.uint8),
                      down_scales=rng.integers(120, 131, (d, f // 32), dtype=np.uint8))
    x = rng.standard_normal((T, d)).astype(np.float32)
    ids = np.stack([np.sort(rng.choice(E, k, replace=False)) for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k))
    ref = np.zeros((T, d))
    for t in range(T):
        for j in range(k):
            ref[t] += w[t, j] * oracle.expert_forward_mxq(exs[int(ids[t, j])], x[t])
    seen = []
    got = oracle.combine_grouped_mxq(x, ids, w, lambda e: exs[e],
                                     on_expert=lambda e, ts, js, h32, Wd: seen.append((e, len(ts), h32.shape)))
    scale = np.abs(ref).max()
    assert np.max(np.abs(got - ref)) <= 1e-12 * scale
    assert sorted(s[0] for s in seen) == sorted(set(int(v) for v in ids.ravel()))
    assert all(s[2] == (s[1], f) for s in seen)
    w2 = w.copy()
    w2[3, 2] = 0.0
    bad = oracle.combine_grouped_mxq(x, ids, w2, lambda e: exs[e])
    assert np.max(np.abs(bad - ref)) > 1e-3 * scale
