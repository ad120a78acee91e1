"""GPU parity of the packed MXFP4 products against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import TOL, Pool, rel_err
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _matmul(packed, scales, x):
    rows, cols = packed.shape[0], packed.shape[1] * 2
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    P, S, X = _dev(packed), _dev(scales), _dev(x.astype(np.float32))
    k.matmul_mxfp4(y, X, P, S, rows, cols)
    torch.cuda.synchronize()
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("rows,cols", [(1, 32), (7, 96), (33, 1024), (130, 1056), (5, 16384),
                                       (1536, 7168), (7168, 1536)])
def test_matmul_mxfp4_vs_oracle(rows, cols):
    packed, scales = synth.matrix(synth.K_GATE_PACKED, synth.K_GATE_SCALES, rows, cols, 3, 1,
                                  rows + cols)
    x = synth.normal_f32((cols,), synth.tag(synth.K_MISC, 3, 1, cols))
    got = _matmul(packed, scales, x)
    ref = oracle.matvec(packed, scales, x.astype(np.float64))
    assert rel_err(got, ref) <= 1e-5  # fp32 accumulation, far inside the 2e-3 bar


def test_decode_bit_exact_all_codes_all_exponents():
    """16 codes x 256 exponents: with a one-hot x the kernel returns the
    decoded weight itself, which must equal the oracle's fp64 value rounded to
    fp32 wherever that is finite."""
    rows = 256
    packed = np.zeros((rows, 16), np.uint8)
    codes = np.array(list(range(16)) * 2)
    for b in range(16):
        packed[:, b] = codes[2 * b] | (codes[2 * b + 1] << 4)
    scales = np.arange(256, dtype=np.uint8).reshape(rows, 1)
    Wd = oracle.dequant(packed, scales)
    for j in range(32):
        x = np.zeros(32, np.float32)
        x[j] = 1.0
        got = _matmul(packed, scales, x)
        want = Wd[:, j].astype(np.float32).astype(np.float64)
        fin = np.isfinite(want) & (np.abs(Wd[:, j]) < 3.4e38)
        assert np.array_equal(got[fin], want[fin]), j
        assert fin.sum() >= 250


def test_nan_scale_and_extreme_exponents():
    rows, cols = 64, 512
    packed, scales = synth.matrix(synth.K_UP_PACKED, synth.K_UP_SCALES, rows, cols, 3, 2, 0)
    scales = scales.copy()
    scales[::3, 1] = 255          # NaN groups contribute nothing
    scales[1::5, 2] = 0           # 2^-127
    scales[2::7, 3] = 140         # large but finite in fp32
    x = synth.normal_f32((cols,), synth.tag(synth.K_MISC, 3, 2, 1))
    got = _matmul(packed, scales, x)
    ref = oracle.matvec(packed, scales, x.astype(np.float64))
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref) <= 1e-5


@pytest.mark.parametrize("d,f", [(96, 64), (1056, 544), (7168, 1536)])
def test_expert_gemv_vs_oracle(d, f):
    """One expert, one token (the single-expert workload at full size)."""
    pool = Pool(0, 0, 2, d, f)
    ws = torch.zeros(k.expert_gemv_workspace(d, f) // 4, dtype=torch.float32, device="cuda")
    for e in range(2):
        x = synth.token_f32(0, e, d)
        y = torch.empty(d, dtype=torch.float32, device="cuda")
        k.expert_gemv(y, torch.from_numpy(x).cuda(), pool.views[e], d, f, ws)
        torch.cuda.synchronize()
        ref = oracle.expert_forward(pool.planes(e), x.astype(np.float64))
        assert rel_err(y.cpu().numpy(), ref) <= TOL


def test_expert_gemv_swapped_nibbles_fail():
    """A nibble-swapped copy of the weights must NOT match: the check is on
    positions, not on value histograms."""
    d, f = 256, 64
    ex = synth.expert(0, 0, 7, d, f)
    sw = dict(ex)
    for kk in ("gate_packed", "up_packed", "down_packed"):
        sw[kk] = ((ex[kk] >> 4) | (ex[kk] << 4)).astype(np.uint8)
    blob = torch.empty(k.expert_bytes(d, f), dtype=torch.uint8, device="cuda")
    k.pack_expert(blob, sw, d, f)
    ws = torch.zeros(k.expert_gemv_workspace(d, f) // 4, dtype=torch.float32, device="cuda")
    x = synth.token_f32(0, 1, d)
    y = torch.empty(d, dtype=torch.float32, device="cuda")
    k.expert_gemv(y, torch.from_numpy(x).cuda(), k.expert_view(blob.data_ptr(), d, f), d, f, ws)
    torch.cuda.synchronize()
    ref = oracle.expert_forward(ex, x.astype(np.float64))
    assert rel_err(y.cpu().numpy(), ref) > 0.1


@pytest.mark.parametrize("d,f", [(512, 512), (1024, 512), (4096, 2048), (7168, 1536), (7168, 2048)])
def test_expert_gemv_repeats_on_one_workspace(d, f):
    """From fewer gate/up stages than CTAs to the full size: three calls in a
    row on one workspace, each against the oracle."""
    pool = Pool(0, 0, 3, d, f)
    ws = torch.zeros(k.expert_gemv_workspace(d, f) // 4, dtype=torch.float32, device="cuda")
    for e in range(3):
        x = synth.token_f32(0, 100 + e, d)
        y = torch.full((d,), float("nan"), dtype=torch.float32, device="cuda")
        k.expert_gemv(y, torch.from_numpy(x).cuda(), pool.views[e], d, f, ws)
        torch.cuda.synchronize()
        ref = oracle.expert_forward(pool.planes(e), x.astype(np.float64))
        assert rel_err(y.cpu().numpy(), ref) <= TOL, (d, f, e)
    assert k.device_error() == 0
