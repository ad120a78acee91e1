"""Pins of the oracle's bf16 shared expert ("kimi-k3-in-c" explainer, "Why
the trunk stays at 16 bits"; two shared experts per layer, "Running Kimi K3
locally", "What are the four reductions, and why is the answer
unchanged?"): bf16 weights read exactly, closed forms with one-hot weights
that tell gate from up and the down direction, a library matrix product on
random shapes, and the sum over the shared experts."""
import math

import numpy as np

import oracle

BF16_ONE, BF16_TWO, BF16_HALF, BF16_MINUS3 = 0x3F80, 0x4000, 0x3F00, 0xC040


def _bf16_bits(a):
    """Round-to-nearest-even bf16 bit patterns of fp32 values (test-side)."""
    u = np.asarray(a, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_values(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_one_hot_closed_form_tells_gate_up_and_down_apart():
    d, f = 64, 32
    gate = np.zeros((f, d), np.uint16)
    up = np.zeros((f, d), np.uint16)
    down = np.zeros((d, f), np.uint16)
    gate[5, 10] = BF16_ONE       # g_5 = x_10
    up[5, 20] = BF16_TWO         # u_5 = 2 x_20
    down[7, 5] = BF16_MINUS3     # y_7 = -3 h_5
    down[9, 5] = BF16_HALF       # y_9 = 0.5 h_5
    x = np.zeros(d)
    x[10], x[20] = 1.5, -0.75
    y = oracle.shared_expert(dict(gate=gate, up=up, down=down), x)
    h5 = 1.5 / (1.0 + math.exp(-1.5)) * (2 * -0.75)
    want = np.zeros(d)
    want[7], want[9] = -3 * h5, 0.5 * h5
    assert np.allclose(y, want, rtol=1e-15, atol=0)
    # swapping gate and up changes the result (silu is not symmetric)
    y2 = oracle.shared_expert(dict(gate=up, up=gate, down=down), x)
    assert not np.allclose(y2, y)


def test_matches_a_library_matrix_product():
    rng = np.random.default_rng(3)
    d, f = 96, 64
    ex = dict(gate=_bf16_bits(rng.standard_normal((f, d)) * 0.1),
              up=_bf16_bits(rng.standard_normal((f, d)) * 0.1),
              down=_bf16_bits(rng.standard_normal((d, f)) * 0.1))
    x = rng.standard_normal(d)
    G, U, D = (_bf16_values(ex[k]) for k in ("gate", "up", "down"))
    g, u = G @ x, U @ x
    want = D @ (g / (1.0 + np.exp(-g)) * u)
    y = oracle.shared_expert(ex, x)
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_forward_sums_the_shared_experts_per_token():
    rng = np.random.default_rng(4)
    d, f, T = 64, 32, 3
    exs = [dict(gate=_bf16_bits(rng.standard_normal((f, d)) * 0.2),
                up=_bf16_bits(rng.standard_normal((f, d)) * 0.2),
                down=_bf16_bits(rng.standard_normal((d, f)) * 0.2)) for _ in range(2)]
    x = rng.standard_normal((T, d))
    out = oracle.shared_forward(x, exs)
    for t in range(T):
        want = oracle.shared_expert(exs[0], x[t]) + oracle.shared_expert(exs[1], x[t])
        assert np.allclose(out[t], want, rtol=1e-14, atol=1e-14 * np.abs(want).max())
    # a planted mistake: one expert counted twice
    bad = oracle.shared_forward(x, [exs[0], exs[0]])
    assert not np.allclose(bad, out)


def test_zero_input_and_bf16_extremes():
    d, f = 32, 32
    ex = dict(gate=np.full((f, d), 0x7F7F, np.uint16),   # largest finite bf16
              up=np.full((f, d), 0x0001, np.uint16),     # smallest subnormal bf16
              down=np.full((d, f), BF16_ONE, np.uint16))
    assert not oracle.shared_expert(ex, np.zeros(d)).any()
    assert abs(oracle.bf16_value(0x7F7F) - 3.3895313892515355e38) < 1e24
    assert oracle.bf16_value(0x0001) == 2.0 ** -133
