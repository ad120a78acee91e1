"""The arithmetic claim under the block-scaled batch-1 path, checked on the
CPU (no GPU): an fp32 32-block written as 16 E2M1 pieces, each with one
power-of-two scale, is reproduced exactly.

Piece p takes the residual r of the pieces before it, picks the smallest
exponent s with 6 * 2^s >= max |r|, rounds |r| / 2^s to the E2M1 magnitudes
{0, .5, 1, 1.5, 2, 3, 4, 6} and subtracts the rounded value.  The steps are
restated here in float32 numpy arithmetic, to show the properties the kernel
relies on: every subtraction is exact in fp32, the residual shrinks by at
least 3x per piece, so 16 pieces leave less than 3^-16 of the block's largest
magnitude, and blocks of Gaussian values come back exactly."""
import numpy as np

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _pieces(block):
    r = np.asarray(block, np.float32).copy()
    out = []
    for _ in range(16):
        m = float(np.max(np.abs(r)))
        if m == 0.0:
            out.append((np.zeros(32), 0))
            continue
        s = int(np.ceil(np.log2(m / 6.0)))  # smallest s with 6 * 2^s >= m
        while 6.0 * 2.0 ** (s - 1) >= m:
            s -= 1
        while 6.0 * 2.0 ** s < m:
            s += 1
        s = min(max(s, -126), 126)
        a = np.abs(r).astype(np.float64) / 2.0 ** s
        code = np.searchsorted(MIDS, a, side="right")  # half-up at a midpoint
        q = (np.sign(r) * GRID[code] * 2.0 ** s).astype(np.float64)
        nr = (r.astype(np.float64) - q)
        # the subtraction is exact in fp32: the fp64 difference is an fp32 value
        assert np.array_equal(nr.astype(np.float32).astype(np.float64), nr)
        if m > 2.0 ** -100:
            assert np.max(np.abs(nr)) <= m / 3.0
        r = nr.astype(np.float32)
        out.append((q, s))
    return out, r


def test_sixteen_pieces_reproduce_gaussian_blocks_exactly():
    """Blocks of N(0, 1) values at any scale of the normal range (zeros
    planted in some) come back exactly."""
    rng = np.random.default_rng(51)
    for trial in range(400):
        k = int(rng.integers(-90, 110))
        b = (rng.standard_normal(32) * 2.0 ** k).astype(np.float32)
        if trial % 2:
            b[rng.integers(0, 32, 6)] = 0.0
        pieces, rest = _pieces(b)
        total = np.sum([q for q, _ in pieces], axis=0)
        assert np.array_equal(total, b.astype(np.float64)), trial
        assert not rest.any()


def test_wide_blocks_stay_within_the_residual_bound():
    """In general the residual after 16 pieces is at most 3^-16 (2.3e-8) of
    the block's largest magnitude: a value far below the block maximum can
    lose its last bits.  Blocks spanning 2^20 in magnitude."""
    rng = np.random.default_rng(53)
    exact = 0
    for trial in range(300):
        k = int(rng.integers(-80, 100))
        b = (rng.standard_normal(32) * 2.0 ** k * 2.0 ** rng.integers(-20, 1, 32)).astype(np.float32)
        pieces, rest = _pieces(b)
        total = np.sum([q for q, _ in pieces], axis=0)
        err = np.max(np.abs(total - b.astype(np.float64)))
        assert err <= np.max(np.abs(b)) * 3.0 ** -16
        exact += err == 0
    assert exact > 250  # most still come back exactly


def test_exact_grid_blocks_need_one_piece():
    """A block already on one E2M1 grid is the first piece; the others are 0."""
    rng = np.random.default_rng(52)
    for s in (-20, 0, 7):
        c = rng.integers(0, 8, 32)
        c[0] = 7
        b = (GRID[c] * np.where(rng.integers(0, 2, 32) == 1, 1, -1) * 2.0 ** s).astype(np.float32)
        pieces, rest = _pieces(b)
        assert np.array_equal(pieces[0][0], b.astype(np.float64))
        assert all(not q.any() for q, _ in pieces[1:])


def test_subnormal_residuals_are_where_exactness_ends():
    """Near the fp32 subnormal range the clamped scale (2^-126) can no longer
    follow the residual down: the pieces then leave a remainder below
    2^-126 * 0.25 per element, which is why the kernel's exactness is stated
    for normal-range blocks."""
    b = np.full(32, np.float32(2.0 ** -120) * np.float32(1.0 + 2.0 ** -23), np.float32)
    pieces, rest = _pieces(b)
    total = np.sum([q for q, _ in pieces], axis=0)
    assert np.max(np.abs(total - b.astype(np.float64))) <= 2.0 ** -128
