"""GPU parity of the block-scaled batch-1 path (K3MOE_OPT_MX): the packed
E2M1 planes and their E8M0 scales feed tcgen05 kind::mxf4 MMAs directly and
the activations become 16 E2M1 pieces per 32-block.  Expected values come
from the fp64 oracle; the fused CUDA-core kernel of the same library is a
second witness."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import TOL, Pool, margin_subs, rel_err, router_tensor, tokens, tokens_device
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _run(L, X, K):
    out = torch.empty((1, L.d), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, K), dtype=torch.int32, device="cuda")
    w = torch.empty((1, K), dtype=torch.float32, device="cuda")
    L.forward(X, 1, out, ids, w)
    torch.cuda.synchronize()
    assert k.device_error() == 0
    return out.cpu().numpy()[0], ids.cpu().numpy()[0], w.cpu().numpy()[0]


def _oracle(pool, Wr_bits, bias, K, xd):
    lg = oracle.router_logits(xd[None], Wr_bits)
    rids, rw, m = oracle.topk(lg, K, None if bias is None else np.asarray(bias, np.float64))
    ref = oracle.combine(xd[None], rids, rw, pool.experts(rids[0]), pool.E)[0]
    return ref, rids[0], rw[0], m[0]


def _case(pool, Wr_bits, bias, K, T, bf16=False, witness=True, seed=None):
    d, f, E = pool.d, pool.f, pool.E
    seed = pool.pool if seed is None else seed
    subs = margin_subs(seed, T, d, Wr_bits, K, bias, bf16=bf16)
    Xd = tokens(seed, np.arange(T), d, subs, bf16)
    X = tokens_device(seed, T, d, subs, bf16)
    bt = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).cuda()
    L = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, bt, max_tokens=1)
    assert L.mx_t1() and not L.fused_t1()
    if witness:
        L2 = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, bt, max_tokens=1)
        L2.set_option(k.K3MOE_OPT_MX, 0)
    for t in range(T):
        out, ids, w = _run(L, X[t:t + 1].contiguous(), K)
        ref, rids, rw, m = _oracle(pool, Wr_bits, bias, K, Xd[t])
        assert m >= 1e-3
        assert np.array_equal(ids, rids)
        assert np.allclose(w, rw, rtol=2e-4, atol=1e-7)
        e = rel_err(out, ref)
        assert e <= TOL, (t, e)
        if witness and not bf16:
            out2, ids2, _ = _run(L2, X[t:t + 1].contiguous(), K)
            assert np.array_equal(ids2, ids)
            assert rel_err(out, out2) <= 1e-5, t
    L.close()
    if witness:
        L2.close()


@pytest.fixture(scope="module")
def mid():
    E, d, f = 48, 1024, 512
    pool = Pool(6, 0, E, d, f)
    return pool, synth.router_bf16(6, 0, E, d), synth.bias_normal(6, 0, E)


@pytest.mark.parametrize("K,use_bias", [(1, False), (8, True), (16, False), (16, True)])
def test_mx_matches_oracle_and_fused_kernel(mid, K, use_bias):
    pool, Wr_bits, bias = mid
    _case(pool, Wr_bits, bias if use_bias else None, K, 3)


def test_mx_bf16_token(mid):
    pool, Wr_bits, bias = mid
    _case(pool, Wr_bits, None, 8, 2, bf16=True)


def test_mx_tiles_split_over_many_ctas():
    """Two experts of d = f = 512: 16 units per phase for 152 CTAs, so most
    CTAs hold no unit and every tile's K steps are spread over CTAs whose
    partial sums meet in the workspace."""
    E, K, d, f = 16, 2, 512, 512
    pool = Pool(16, 0, E, d, f)
    _case(pool, synth.router_bf16(16, 0, E, d), None, K, 3)


def test_mx_scales_outside_the_f16_range():
    """E8M0 bytes in [100, 150]: the hardware applies any scale."""
    E, K, d, f = 32, 4, 1024, 512
    pool = Pool(17, 0, E, d, f, e_lo=100, e_hi=150)
    _case(pool, synth.router_bf16(17, 0, E, d), None, K, 3)


def test_mx_nan_scale_groups_are_dropped():
    """Scale byte 255 in every third group of some gate, up and down rows of
    every expert: those groups contribute nothing, as in the oracle."""
    E, K, d, f = 16, 4, 1024, 512
    pool = Pool(18, 0, E, d, f)
    for e in range(E):
        planes = pool.planes(e)
        planes["gate_scales"][:64, ::3] = 255
        planes["up_scales"][100:130, 1::5] = 255
        planes["down_scales"][::7, ::4] = 255
        k.pack_expert(pool.blobs[e], planes, d, f)
        pool.override[e] = planes
    torch.cuda.synchronize()
    _case(pool, synth.router_bf16(18, 0, E, d), None, K, 3)


def test_mx_repeats_and_resets_its_counters(mid):
    """Repeated forwards of one token agree to fp32 rounding (the order of the
    k experts' additions into the output is not fixed), and the cross-CTA
    counters are back to zero after every launch (a stale count would let a
    later launch read h pieces before they are written)."""
    pool, Wr_bits, bias = mid
    K, d = 16, pool.d
    subs = margin_subs(6, 1, d, Wr_bits, K)
    X = tokens_device(6, 1, d, subs)
    L = k.Layer(pool.E, K, d, pool.f, router_tensor(Wr_bits), pool.views, max_tokens=1)
    first, _, _ = _run(L, X, K)
    for _ in range(6):
        again, _, _ = _run(L, X, K)
        assert rel_err(again, first) <= 1e-6
    L.close()


def test_mx_full_shape_with_bias():
    """d = 7168, f = 1536, 64 experts, top-16, a selection bias."""
    E, K, d, f = 64, 16, 7168, 1536
    pool = Pool(19, 0, E, d, f)
    _case(pool, synth.router_bf16(19, 0, E, d), synth.bias_normal(19, 0, E), K, 2)
