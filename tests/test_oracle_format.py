"""Pins of the oracle's MXFP4 decode and packed product against what the pages
and the mathematics fix (no GPU).

Each test is built so that a plausible mistake in the oracle fails it: a wrong
table entry, the nibble order reversed, the scale of the wrong group, a NaN
scale read as 2^128, a transposed product, or a group-wise reordering that
changes more than rounding.
"""
import math

import numpy as np
import pytest

import oracle


def _bitfield_e2m1(code):
    """E2M1 from its bit fields, written independently of any table:
    s = bit 3, E = bits 2..1, m = bit 0; E == 0 is subnormal (m * 0.5),
    otherwise (1 + m/2) * 2^(E-1)."""
    s = (code >> 3) & 1
    E = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if E == 0 else (1.0 + m / 2.0) * 2.0 ** (E - 1)
    return -mag if s else mag


def test_e2m1_table_matches_bit_fields():
    for c in range(16):
        assert oracle.e2m1_value(c) == _bitfield_e2m1(c), c
    # the largest magnitude is 6 and code 8 is a (negative) zero
    assert oracle.e2m1_value(7) == 6.0 and oracle.e2m1_value(15) == -6.0
    assert oracle.e2m1_value(8) == 0.0 and math.copysign(1.0, oracle.e2m1_value(8)) == -1.0


def test_e8m0_values():
    for e in range(255):
        assert oracle.e8m0_value(e) == 2.0 ** (e - 127)
    assert math.isnan(oracle.e8m0_value(255))


def test_decode_enumerates_all_codes_and_exponents():
    """All 16 codes x all 256 exponents through the oracle's dequantiser.
    Row e holds exponent e; its 32 weights are codes 0..15 twice (low nibble
    even index).  Exponent 255 must zero the group."""
    rows = 256
    packed = np.zeros((rows, 16), np.uint8)
    codes = np.array(list(range(16)) * 2)
    for b in range(16):
        packed[:, b] = codes[2 * b] | (codes[2 * b + 1] << 4)
    scales = np.arange(256, dtype=np.uint8).reshape(rows, 1)
    W = oracle.dequant(packed, scales)
    for e in range(256):
        for j in range(32):
            want = 0.0 if e == 255 else _bitfield_e2m1(codes[j]) * 2.0 ** (e - 127)
            assert W[e, j] == want, (e, j)


def test_nibble_order_low_is_even():
    """The low nibble is the even-index weight ("Running Kimi K3 locally",
    four reductions).  0x21: element 0 = code 1 (0.5), element 1 = code 2 (1.0)."""
    packed = np.array([[0x21] + [0] * 15], np.uint8)
    scales = np.array([[127]], np.uint8)
    W = oracle.dequant(packed, scales)
    assert W[0, 0] == 0.5 and W[0, 1] == 1.0 and not W[0, 2:].any()
    x = np.zeros(32)
    x[0] = 1.0
    assert oracle.matvec(packed, scales, x)[0] == 0.5
    x[:] = 0
    x[1] = 1.0
    assert oracle.matvec(packed, scales, x)[0] == 1.0


def test_swapped_nibbles_same_histogram_different_product():
    """Swapping the nibbles keeps every value histogram but moves weights: a
    check on distributions would pass, a check on positions must not
    ("kimi-k3-in-c: A 176 KB Engine...", 'What byte-identical actually costs')."""
    rng = np.random.default_rng(7)
    packed = rng.integers(0, 256, (8, 64), dtype=np.uint8)
    scales = rng.integers(120, 131, (8, 4), dtype=np.uint8)
    swapped = ((packed >> 4) | (packed << 4)).astype(np.uint8)
    A = oracle.dequant(packed, scales)
    B = oracle.dequant(swapped, scales)
    assert np.array_equal(np.sort(A, axis=None), np.sort(B, axis=None))
    x = rng.standard_normal(128)
    assert not np.allclose(oracle.matvec(packed, scales, x), oracle.matvec(swapped, scales, x))


def test_nan_scale_zeroes_only_its_group():
    """E8M0 byte 255 is NaN; its 32 weights contribute nothing and the rest of
    the row is untouched (176 KB Engine, 'What byte-identical actually costs';
    explainer 'Reduction one')."""
    packed = np.full((1, 48), 0x77, np.uint8)  # every weight code 7 = 6.0
    scales = np.array([[127, 255, 128]], np.uint8)
    x = np.ones(96)
    y = oracle.matvec(packed, scales, x)[0]
    assert y == 32 * 6.0 * 1.0 + 32 * 6.0 * 2.0
    assert oracle.matvec_groupwise(packed, scales, x)[0] == y
    # a NaN scale read as 2^128 would add 32*6*2^128
    assert y < 1e30


def test_group_scale_index_and_orientation_one_hot():
    """Row r holds a single 1.0 (code 2) at column c_r inside group c_r // 32,
    whose exponent is 127 + g: y[r] = 2^g * x[c_r].  Catches a transposed
    product, a wrong group-scale index and an off-by-one column."""
    rows, cols = 6, 128
    cs = [0, 33, 64, 127, 95, 1]
    packed = np.zeros((rows, cols // 2), np.uint8)
    for r, c in enumerate(cs):
        packed[r, c // 2] = 2 << (4 * (c & 1))
    scales = np.tile(np.array([127, 128, 129, 130], np.uint8), (rows, 1))
    x = np.arange(1, cols + 1, dtype=np.float64) * 0.25
    y = oracle.matvec(packed, scales, x)
    for r, c in enumerate(cs):
        assert y[r] == 2.0 ** (c // 32) * x[c]


def test_constant_matrix_closed_form():
    """All weights code 5 (3.0) with exponent 127 + 2: y = 12 * sum(x)."""
    packed = np.full((3, 32), 0x55, np.uint8)
    scales = np.full((3, 2), 129, np.uint8)
    x = np.linspace(-1, 2, 64)
    y = oracle.matvec(packed, scales, x)
    assert np.all(np.abs(y - 12.0 * x.sum()) <= 1e-13 * np.abs(x).sum() * 12)


@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 64), (8, 128), (5, 96)])
def test_groupwise_order_matches_definition(rows, cols):
    """The pages' group-wise order equals dequantise-then-multiply up to
    rounding: products are exact in double, so the two sums differ by about
    one double ulp (explainer, 'A floating-point contract').  Bound checked:
    1e-12 of sum |w x| (the pages' own gate is 1e-6)."""
    rng = np.random.default_rng(rows * 1000 + cols)
    for trial in range(20):
        packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
        scales = rng.integers(100, 150, (rows, cols // 32), dtype=np.uint8)
        if trial == 0:  # every code appears
            packed.flat[:8] = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]
        x = rng.standard_normal(cols).astype(np.float32).astype(np.float64)
        a = oracle.matvec(packed, scales, x)
        b = oracle.matvec_groupwise(packed, scales, x)
        mag = np.abs(oracle.dequant(packed, scales)) @ np.abs(x)
        assert np.all(np.abs(a - b) <= 1e-12 * mag + 1e-300)


def test_matvec_exact_on_dyadic_inputs():
    """With x on a dyadic grid every partial sum is exact in double, so the
    fp64 product must equal integer arithmetic on (2 * E2M1) codes exactly."""
    rng = np.random.default_rng(3)
    rows, cols = 7, 96
    packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    scales = np.full((rows, cols // 32), 127, np.uint8)
    xi = rng.integers(-64, 65, cols)
    x = xi.astype(np.float64) / 8.0
    y = oracle.matvec(packed, scales, x)
    # integer decode written from the bit fields: 2*value is an integer
    twice = {c: int(round(2 * _bitfield_e2m1(c))) for c in range(16)}
    for r in range(rows):
        acc = 0
        for j in range(cols):
            b = int(packed[r, j // 2])
            c = (b >> 4) if (j & 1) else (b & 15)
            acc += twice[c] * int(xi[j])
        assert y[r] == acc / 16.0


def test_byte_arithmetic_matches_pages(golden):
    d, f = 7168, 1536
    assert golden["hidden_size"]["value"] == d
    assert 3 * d * f == golden["expert_params"]["value"]
    assert oracle.expert_bytes(d, f) == golden["expert_bytes"]["value"]
    assert oracle.matrix_bytes(f, d) == 5505024 + 344064 == 5849088
    assert oracle.expert_bytes(d, f) / (3 * d * f) == golden["bytes_per_weight"]["value"]
    assert 4 / 8 + 8 / (8 * golden["group_size"]["value"]) == golden["bytes_per_weight"]["value"]
    per_token = golden["experts_per_token"]["value"] * oracle.expert_bytes(d, f)
    assert per_token == 25829572608
    assert round(per_token / 1e9, 2) == golden["packed_gb_per_token"]["value"]
    fp32 = 3 * d * f * 4
    assert round(fp32 / 1e6) == golden["fp32_expert_mb"]["value"]
    assert round(golden["experts_per_token"]["value"] * fp32 / 1e9) == golden["dequant_gb_per_token"]["value"]
    pool = golden["routed_experts_total"]["value"] * oracle.expert_bytes(d, f)
    assert pool == 1446456066048
    assert abs(pool / 1e12 - golden["routed_pool_tb_printed"]["value"]) < 1.5e-3
    assert golden["routed_experts_total"]["value"] == 92 * golden["experts_per_layer"]["value"]
