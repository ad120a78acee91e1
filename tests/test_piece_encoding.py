"""The arithmetic claim under the block-scaled batch-1 path, checked on the
CPU (no GPU): an fp32 32-block written as 16 E2M1 pieces, each with one
power-of-two scale, is reproduced to 2^-32 of the block's scale, and exactly
for every value within 2^8 of the block's largest magnitude.

The rule, restated here with integer arithmetic in numpy: E is the biased
exponent of the block's largest magnitude (at least 1); each |v| becomes the
32-bit integer M = |v| * 2^(158 - E), rounded to the nearest integer (ties
up) where it is not one already; piece p is the p-th base-4 digit of M from
the top, d_p = (M >> (30 - 2p)) & 3, taken as the E2M1 magnitude d_p / 2
(codes 0-3) with the sign of v, scaled by 2^(E - 127 - 2p); a piece whose
scale byte E - 2p would be negative is left out.  So the pieces add up to
sign * M * 2^(E - 158)."""
import numpy as np

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _pieces(block):
    """Returns (codes [16][32], scale bytes [16]) of one fp32 block."""
    b = np.asarray(block, np.float32)
    bits = b.view(np.uint32).astype(np.int64)
    ab = bits & 0x7FFFFFFF
    assert np.all(ab < 0x7F800000)
    mb = int(ab.max())
    codes = np.zeros((16, 32), np.int64)
    if mb == 0:
        return codes, np.full(16, 127, np.int64)
    E = max(mb >> 23, 1)
    ev = np.maximum(ab >> 23, 1)
    m24 = (ab & 0x7FFFFF) | np.where((ab >> 23) > 0, 0x800000, 0)
    sh = ev - E + 8
    M = np.zeros(32, np.int64)
    for i in range(32):
        if sh[i] >= 0:
            M[i] = int(m24[i]) << int(sh[i])
        elif -sh[i] < 32:
            M[i] = (int(m24[i]) + (1 << int(-sh[i] - 1))) >> int(-sh[i])
    assert np.all(M < 2 ** 32)
    scales = np.array([max(E - 2 * p, 0) for p in range(16)], np.int64)
    for p in range(16):
        if E - 2 * p < 0:
            continue
        d = (M >> (30 - 2 * p)) & 3
        codes[p] = d | np.where(bits >> 31, 8, 0)
    return codes, scales


def _value(codes, scales):
    """Sum of the pieces in fp64 (every term and partial sum is exact there)."""
    mag = GRID[codes & 7]
    sign = np.where(codes & 8, -1.0, 1.0)
    return np.sum(sign * mag * (2.0 ** (scales.astype(np.float64) - 127))[:, None], axis=0)


def _e(block):
    return max(int(np.max(np.abs(np.asarray(block, np.float32)).view(np.uint32))) >> 23, 1)


def test_values_within_two_to_the_eight_of_the_maximum_are_exact():
    """Blocks of N(0, 1) values at any scale of the normal range (zeros
    planted in some): every value at least 2^-8 of the block's scale comes
    back exactly, the rest within half a unit of M."""
    rng = np.random.default_rng(51)
    for trial in range(400):
        k = int(rng.integers(-90, 110))
        b = (rng.standard_normal(32) * 2.0 ** k).astype(np.float32)
        if trial % 2:
            b[rng.integers(0, 32, 6)] = 0.0
        codes, scales = _pieces(b)
        got = _value(codes, scales)
        E = _e(b)
        ref = b.astype(np.float64)
        big = np.abs(ref) >= 2.0 ** (E - 135)
        assert np.array_equal(got[big], ref[big]), trial
        assert np.all(np.abs(got - ref) <= 2.0 ** (E - 159)), trial


def test_wide_blocks_stay_within_two_to_the_minus_32_of_the_block_scale():
    """Blocks spanning 2^40 in magnitude: the error of every value is at most
    2^(E - 159), that is 2^-32 of 2^(E - 127), the block's scale."""
    rng = np.random.default_rng(53)
    for trial in range(300):
        k = int(rng.integers(-60, 100))
        b = (rng.standard_normal(32) * 2.0 ** k * 2.0 ** rng.integers(-40, 1, 32)).astype(np.float32)
        codes, scales = _pieces(b)
        E = _e(b)
        err = np.max(np.abs(_value(codes, scales) - b.astype(np.float64)))
        assert err <= 2.0 ** (E - 159), trial
        assert err <= np.max(np.abs(b.astype(np.float64))) * 2.0 ** -31


def test_digits_sit_in_the_pieces_of_their_weight():
    """1.5 * 2^e (the block maximum) is piece 0 alone (code 3); adding 2^(e-2)
    (one unit of digit 1) sets piece 1 to code 2 (value 1 at scale 2^(e-2))."""
    for e in (-20, 0, 37):
        b = np.zeros(32, np.float32)
        b[0] = np.float32(1.5 * 2.0 ** e)
        b[1] = np.float32(-(1.5 * 2.0 ** e + 2.0 ** (e - 2)))
        codes, scales = _pieces(b)
        E = e + 127
        assert scales[0] == E and scales[1] == E - 2
        assert codes[0, 0] == 3 and not codes[1:, 0].any()
        assert codes[0, 1] == 3 | 8 and codes[1, 1] == 2 | 8 and not (codes[2:, 1] & 7).any()
        assert np.array_equal(_value(codes, scales), b.astype(np.float64))


def test_tiny_blocks_leave_out_the_pieces_below_the_scale_range():
    """When E < 30 the pieces whose byte E - 2p would be negative are left
    out (scale byte 0, code 0 or -0): what they would have carried is below
    2^-126, and the rest is still exact to 2^(E - 159) or to the first left-out
    digit, whichever is larger."""
    rng = np.random.default_rng(54)
    for E in (1, 2, 7, 20, 29):
        for trial in range(20):
            mant = rng.uniform(1.0, 2.0, 32)
            b = (mant * 2.0 ** (max(E, 1) - 127) * rng.choice([-1, 1], 32)).astype(np.float32)
            codes, scales = _pieces(b)
            assert _e(b) == E
            pmax = E // 2
            assert np.all(scales[pmax + 1:] == 0) and not (codes[pmax + 1:] & 7).any()
            err = np.max(np.abs(_value(codes, scales) - b.astype(np.float64)))
            assert err <= max(2.0 ** (E - 159), 2.0 ** (E - 127 - 2 * pmax))


def test_subnormal_blocks():
    """A block of subnormal values (E = 1): piece 0 alone, M = mantissa * 2^8,
    so the value m * 2^-149 keeps its top two bits."""
    b = (np.arange(32, dtype=np.float64) * 2.0 ** -140).astype(np.float32)
    codes, scales = _pieces(b)
    assert _e(b) == 1 and scales[0] == 1
    err = np.max(np.abs(_value(codes, scales) - b.astype(np.float64)))
    assert err < 2.0 ** -126
