"""GPU parity of the tensor-core grouped path (K3MOE_OPT_TC): multi-token
layers whose expert products run as tcgen05 MMAs on exactly decoded bf16
weights.  Expected values come from the fp64 oracle; the CUDA-core grouped
path of the same library is compared as a second witness."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import (TOL, Pool, batch_errors, margin_subs, rel_err, report, router_tensor, tokens,
                         tokens_device)
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _forward(L, X, T, K, tc=True, e4m3=True):
    L.set_option(k.K3MOE_OPT_TC, 1 if tc else 0)
    L.set_option(k.K3MOE_OPT_TC_E4M3, 1 if e4m3 else 0)
    out = torch.empty((T, L.d), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    L.forward(X, T, out, ids, w)
    torch.cuda.synchronize()
    assert k.device_error() == 0
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _case(pool, Wr_bits, bias, K, T, bf16, witness=True, e4m3=True):
    d, f, E = pool.d, pool.f, pool.E
    subs = margin_subs(pool.pool, T, d, Wr_bits, K, bias, bf16=bf16)
    Xd = tokens(pool.pool, np.arange(T), d, subs, bf16)
    X = tokens_device(pool.pool, T, d, subs, bf16)
    bt = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    L = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, bt, max_tokens=T)
    out, ids, w = _forward(L, X, T, K, tc=True, e4m3=e4m3)
    lg = oracle.router_logits(Xd, Wr_bits)
    rids, rw, m = oracle.topk(lg, K, None if bias is None else np.asarray(bias, np.float64))
    assert np.all(m >= 1e-3)
    assert np.array_equal(ids, rids)
    ref = oracle.combine_grouped(Xd, rids, rw, pool.planes)
    norm, elem = batch_errors(out, ref)
    report("tensor path T=%d %s %s" % (T, "bf16" if bf16 else "fp32", "e4m3" if e4m3 else "bf16-kind"),
           norm, elem)
    bad = np.nonzero(norm > TOL)[0]
    assert bad.size == 0, [(int(t), float(norm[t])) for t in bad[:10]]
    if witness:
        out2, ids2, _ = _forward(L, X, T, K, tc=False)
        assert np.array_equal(ids2, ids)
        for t in range(T):
            assert rel_err(out[t], out2[t]) <= 1e-4, t
    L.close()
    return out, ids


@pytest.fixture(scope="module")
def small():
    E, K, d, f = 64, 8, 512, 256
    pool = Pool(5, 0, E, d, f)
    return pool, synth.router_bf16(5, 0, E, d), synth.bias_normal(5, 0, E), K


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("T,bf16,use_bias", [(2, False, False), (37, False, True), (37, True, False),
                                             (200, True, True), (200, False, False)])
def test_tc_small_layer(small, T, bf16, use_bias, e4m3):
    pool, Wr_bits, bias, K = small
    _case(pool, Wr_bits, bias if use_bias else None, K, T, bf16, e4m3=e4m3)


@pytest.fixture(scope="module")
def few_experts():
    """8 experts, top-2: ~150 tokens per expert at T = 600, more than one
    tile of 64 (fp32) or 128 (bf16) tokens."""
    E, K, d, f = 8, 2, 512, 512
    pool = Pool(12, 0, E, d, f)
    return pool, synth.router_bf16(12, 0, E, d), K


@pytest.mark.parametrize("e4m3", [True, False])
@pytest.mark.parametrize("bf16", [False, True])
def test_tc_several_tiles_per_expert(few_experts, bf16, e4m3):
    pool, Wr_bits, K = few_experts
    out, ids = _case(pool, Wr_bits, None, K, 600, bf16, e4m3=e4m3)
    counts = np.bincount(ids.ravel(), minlength=pool.E)
    assert counts.max() > 128


def test_tc_scales_outside_the_f16_range():
    """E8M0 bytes in [100, 150]: groups below 113 or above 142 take the
    general (fp32) decode, the others the f16 one."""
    E, K, d, f = 16, 4, 512, 256
    pool = Pool(13, 0, E, d, f, e_lo=100, e_hi=150)
    _case(pool, synth.router_bf16(13, 0, E, d), None, K, 24, False)


def test_tc_nan_scale_groups_are_dropped():
    """Scale byte 255 in every third gate group of expert 0's first 64 rows:
    those groups contribute 0 on both paths and in the oracle."""
    E, K, d, f = 16, 4, 512, 256
    pool = Pool(14, 0, E, d, f)
    planes = pool.planes(0)
    planes["gate_scales"][:64, ::3] = 255
    k.pack_expert(pool.blobs[0], planes, d, f)
    torch.cuda.synchronize()
    pool.override[0] = planes
    _case(pool, synth.router_bf16(14, 0, E, d), None, K, 40, False)


def test_tc_full_shape_small_batch():
    """d = 7168, f = 1536, 64 experts, top-16, 5 fp32 tokens (tiles of one or
    two tokens, N = 16 columns)."""
    E, K, d, f = 64, 16, 7168, 1536
    pool = Pool(15, 0, E, d, f)
    _case(pool, synth.router_bf16(15, 0, E, d), None, K, 5, False)


def test_tc_layer_forward_twice_is_repeatable(small):
    """The grouped path keeps no state between calls: two forwards of the
    same tokens agree (to the atomic-add summation order)."""
    pool, Wr_bits, bias, K = small
    T, d = 48, pool.d
    subs = margin_subs(5, T, d, Wr_bits, K)
    X = tokens_device(5, T, d, subs)
    L = k.Layer(pool.E, K, d, pool.f, router_tensor(Wr_bits), pool.views, max_tokens=64)
    a, ia, _ = _forward(L, X, T, K)
    b, ib, _ = _forward(L, X, T, K)
    assert np.array_equal(ia, ib)
    for t in range(T):
        assert rel_err(a[t], b[t]) <= 1e-6
    L.close()


def test_e4m3_path_agrees_with_the_bf16_path_and_is_chosen_only_where_exact(small):
    """The two operand kinds of the tensor path give the same outputs to
    fp32-class error on an eligible layer (scale bytes in [120, 130])."""
    pool, Wr_bits, bias, K = small
    T, d = 96, pool.d
    subs = margin_subs(5, T, d, Wr_bits, K)
    X = tokens_device(5, T, d, subs)
    L = k.Layer(pool.E, K, d, pool.f, router_tensor(Wr_bits), pool.views, max_tokens=T)
    a, ia, _ = _forward(L, X, T, K, e4m3=True)
    b, ib, _ = _forward(L, X, T, K, e4m3=False)
    assert np.array_equal(ia, ib)
    for t in range(T):
        assert rel_err(a[t], b[t]) <= 2e-4, t
    L.close()
