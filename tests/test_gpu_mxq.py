"""GPU parity of the MXFP4-activation path (K3MOE_OPT_MXQ): the OCP MX
conversion on the device against the oracle's, code for code; multi-token
layers whose expert products run as block-scaled E2M1 x E2M1 MMAs against
the oracle's mode-B layer, with the tolerance of rounding decisions stated
in the design notes (fp32 gate plus, only where the oracle's h lies within
reach of fp32 rounding of a decision, the change that decision can make).
The error against the exact (unquantised) oracle is reported."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import (Pool, batch_errors, margin_subs, mxq_check, mxq_reference, report, router_tensor,
                         tokens, tokens_device)
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _device_quantize(x):
    """k3moe_mx_quantize of a [rows, cols] tensor -> (codes [rows, cols] as
    4-bit values, scale bytes [rows, cols/32])."""
    rows, cols = x.shape
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device="cuda")
    k.mx_quantize(codes, scales, x, rows, cols)
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    unpacked = np.empty((rows, cols), np.uint8)
    unpacked[:, 0::2] = c & 15
    unpacked[:, 1::2] = c >> 4
    return unpacked, scales.cpu().numpy()


def _edge_rows(rng):
    """Blocks on every rounding midpoint at several exponents, ties, zeros,
    negative zeros, subnormals, huge values, saturation, and non-finite."""
    rows = []
    for ex in (-130, -20, -1, 0, 1, 5, 60, 125):
        s = 2.0 ** ex
        for mids in ([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], [0.5, 1, 1.5, 2, 3, 4, 6, 5.5]):
            v = np.array(mids * 4, np.float64) * s
            v[1::3] *= -1
            v[0] = 6.0 * s  # sets the block maximum, so the scale is 2^ex
            rows.append(v)
    rows.append(np.zeros(32))
    rows.append(-np.zeros(32))
    rows.append(np.full(32, 1e-40) * np.arange(1, 33))  # subnormal fp32
    rows.append(np.linspace(-3e38, 3e38, 32))
    b = rng.standard_normal(32)
    b[7] = np.inf
    rows.append(b)
    b = rng.standard_normal(32)
    b[3] = np.nan
    rows.append(b)
    b = rng.standard_normal(32) * 100
    b[0] = 7.99999  # just below a power of two: amax near the boundary
    rows.append(b)
    return np.concatenate(rows).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_device_quantiser_matches_the_oracle_code_for_code(dtype):
    rng = np.random.default_rng(5)
    rand = (rng.standard_normal(32 * 4096) * np.exp(rng.uniform(-30, 30, 32 * 4096).repeat(1)[:32 * 4096])
            ).astype(np.float32)
    x = np.concatenate([_edge_rows(rng), rand]).astype(np.float32)
    if dtype == "bf16":
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        x = (bits.astype(np.uint32) << 16).view(np.float32)  # the values the device sees
        xt = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        xt = torch.from_numpy(x).cuda()
    cols = 256
    n = (x.size // cols) * cols
    x, xt = x[:n], xt[:n]
    codes, scales = _device_quantize(xt.reshape(-1, cols))
    _, rcodes, rscales = oracle.mx_quantize(x)
    assert np.array_equal(scales.ravel(), rscales)
    ok = rscales.repeat(32) != 255  # codes of a non-finite block are 0 on both sides
    assert np.array_equal(codes.ravel()[ok], rcodes[ok])
    assert np.all(codes.ravel()[~ok] == 0)


def _layer_case(pool, Wr_bits, bias, K, T, bf16, name):
    d, f, E = pool.d, pool.f, pool.E
    subs = margin_subs(pool.pool, T, d, Wr_bits, K, bias, bf16=bf16)
    Xd = tokens(pool.pool, np.arange(T), d, subs, bf16)
    X = tokens_device(pool.pool, T, d, subs, bf16)
    bt = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    L = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, bt, max_tokens=T)
    L.set_option(k.K3MOE_OPT_MXQ, 1)
    assert L.mxq()
    out = torch.empty((T, d), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    L.forward(X, T, out, ids, w)
    torch.cuda.synchronize()
    assert k.device_error() == 0
    out, ids, w = out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()
    lg = oracle.router_logits(Xd, Wr_bits)
    rids, rw, m = oracle.topk(lg, K, None if bias is None else np.asarray(bias, np.float64))
    assert np.array_equal(ids, rids)
    assert np.allclose(w, rw, rtol=2e-4, atol=1e-7)
    ref, bound = mxq_reference(Xd, rids, rw, pool.planes)
    mxq_check(out, ref, bound, name)
    L.close()
    return out, Xd, rids, rw


@pytest.fixture(scope="module")
def small():
    E, K, d, f = 32, 4, 1024, 512
    pool = Pool(41, 0, E, d, f)
    return pool, synth.router_bf16(41, 0, E, d), synth.bias_normal(41, 0, E), K


@pytest.mark.parametrize("T,bf16,use_bias", [(2, False, False), (37, True, True), (300, True, False),
                                             (300, False, True)])
def test_mxq_layer_matches_the_mode_b_oracle(small, T, bf16, use_bias):
    """Tiles of 1..128 tokens (and experts over several tiles at T = 300,
    about 37 tokens per expert on average, more on the biased ones)."""
    pool, Wr_bits, bias, K = small
    _layer_case(pool, Wr_bits, bias if use_bias else None, K, T, bf16,
                "mxq T=%d %s%s" % (T, "bf16" if bf16 else "fp32", " biased" if use_bias else ""))


def test_mxq_experts_over_many_tiles():
    """4 experts, top-2, 700 tokens: about 350 tokens per expert (3 tiles of
    128 and a ragged one); d, f at their smallest block-scaled sizes."""
    E, K, d, f = 4, 2, 512, 512
    pool = Pool(42, 0, E, d, f)
    out, Xd, rids, rw = _layer_case(pool, synth.router_bf16(42, 0, E, d), None, K, 700, True, "mxq 4 experts T=700")
    assert np.bincount(rids.ravel(), minlength=E).max() > 256


def test_mxq_nan_scale_weight_groups_are_dropped():
    """Weight groups with scale byte 255 contribute nothing on the device, as
    in the oracle (the A scale becomes 2^-127)."""
    E, K, d, f = 8, 2, 512, 512
    pool = Pool(43, 0, E, d, f)
    for e in range(E):
        planes = pool.planes(e)
        planes["gate_scales"][:40, ::3] = 255
        planes["down_scales"][::5, 1::4] = 255
        k.pack_expert(pool.blobs[e], planes, d, f)
        pool.override[e] = planes
    torch.cuda.synchronize()
    _layer_case(pool, synth.router_bf16(43, 0, E, d), None, K, 64, False, "mxq nan groups")


D, F, E896, K16 = 7168, 1536, 896, 16


def test_mxq_full_prefill_4096_bf16_biased():
    """The prefill workload: 896 experts, 4096 bf16 tokens, selection bias
    ~ N(0,1); every output vector against the mode-B oracle, the error
    against the exact oracle reported on the first 256 tokens."""
    pool = Pool(1, 0, E896, D, F)
    Wr_bits = synth.router_bf16(1, 0, E896, D)
    bias = synth.bias_normal(1, 0, E896)
    out, Xd, rids, rw = _layer_case(pool, Wr_bits, bias, K16, 4096, True, "mxq prefill T=4096")
    n = 256
    exact = oracle.combine_grouped(Xd[:n], rids[:n], rw[:n], pool.planes)
    norm, elem = batch_errors(out[:n], exact)
    report("mxq prefill T=4096 vs exact oracle (quantisation error, not gated)", norm, elem)
    assert np.all(np.isfinite(out))
