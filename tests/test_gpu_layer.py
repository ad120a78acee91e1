"""GPU parity of the routed-expert layer (router, top-k, experts, combine)
against the fp64 oracle: ids bit-exact on margin-checked tokens, combine
weights and outputs within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import (TOL, Pool, batch_errors, margin_subs, rel_err, report, router_tensor,
                         tokens, tokens_device)
from mxfp4_routed_expert_select_gb300 import k3moe as k

pytestmark = pytest.mark.gpu


def _run(layer, X, T, K):
    out = torch.empty((T, layer.d), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    layer.forward(X, T, out, ids, w)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _check(pool, Wr_bits, bias, K, Xd, out, ids, w, h_bf16=False, name=None):
    """Ids bit-exact and weights close for every token; every output vector
    against the oracle (grouped by expert when the batch is large), gated on
    the normwise error, the per-element error reported."""
    T = Xd.shape[0]
    lg = oracle.router_logits(Xd, Wr_bits)
    rids, rw, m = oracle.topk(lg, K, None if bias is None else bias.astype(np.float64))
    assert np.all(m >= 1e-3)
    assert np.array_equal(ids, rids)
    # fp32 logits over d terms carry ~1e-5 absolute error; w inherits it
    assert np.allclose(w, rw, rtol=2e-4, atol=1e-7)
    if T * K <= 64:
        ref = oracle.combine(Xd, rids, rw, pool.experts(rids), pool.E, h_bf16)
    else:
        ref = oracle.combine_grouped(Xd, rids, rw, pool.planes, h_bf16)
    norm, elem = batch_errors(out, ref)
    if name:
        report(name, norm, elem)
    bad = np.nonzero(norm > TOL)[0]
    assert bad.size == 0, [(int(t), float(norm[t])) for t in bad[:10]]
    return norm, elem


# ------------------------------------------------------------ small layers

@pytest.fixture(scope="module")
def small():
    E, K, d, f = 64, 8, 512, 256
    pool = Pool(5, 0, E, d, f)
    Wr_bits = synth.router_bf16(5, 0, E, d)
    bias = synth.bias_normal(5, 0, E)
    return pool, Wr_bits, bias, E, K, d, f


@pytest.mark.parametrize("T,bf16,use_bias", [(1, False, False), (1, False, True), (1, True, False),
                                             (3, False, False), (17, True, True),
                                             (64, False, False)])
def test_small_layer(small, T, bf16, use_bias):
    pool, Wr_bits, bias, E, K, d, f = small
    b = bias if use_bias else None
    subs = margin_subs(5, T, d, Wr_bits, K, b, bf16=bf16)
    Xd = tokens(5, np.arange(T), d, subs, bf16)
    X = tokens_device(5, T, d, subs, bf16)
    L = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views,
                None if b is None else torch.from_numpy(b).cuda(), max_tokens=max(T, 64))
    out, ids, w = _run(L, X, T, K)
    _check(pool, Wr_bits, b, K, Xd, out, ids, w)
    L.close()


def test_ties_go_to_lower_ids_and_bias_only_selects(small):
    """W_r = 0: every logit is 0, the k lowest ids win with equal weights.
    With a bias that favours the top ids, those are chosen, but the weights
    stay the softmax of the (equal) unbiased logits."""
    pool, Wr_bits, bias, E, K, d, f = small
    zero = torch.zeros((E, d), dtype=torch.int16, device="cuda")
    X = tokens_device(5, 1, d, [0])
    L = k.Layer(E, K, d, f, zero, pool.views, max_tokens=1)
    out, ids, w = _run(L, X, 1, K)
    assert list(ids[0]) == list(range(K)) and np.allclose(w, 1.0 / K)
    bb = torch.from_numpy(np.arange(E, dtype=np.float32)).cuda()
    L2 = k.Layer(E, K, d, f, zero, pool.views, bb, max_tokens=1)
    out, ids, w = _run(L2, X, 1, K)
    assert list(ids[0]) == list(range(E - K, E)) and np.allclose(w, 1.0 / K)
    L.close()
    L2.close()


@pytest.mark.parametrize("path,T", [("mx", 1), ("fused", 1), ("unfused", 1), ("unfused", 5)])
def test_ties_at_the_selection_boundary(fusable, path, T):
    """W_r = 0 and a bias with K-2 distinct high values, then four equal ones
    for the last two slots: the two lowest ids of the tied four are chosen,
    on the block-scaled and the fused batch-1 paths, the batch-1 router and
    the multi-token one.  The expected ids come from the oracle's rule."""
    pool, _, _, E, d, f = fusable
    K = 8
    b = np.zeros(E, np.float32)
    hi = [40, 3, 17, 29, 8, 44]          # K - 2 clear winners
    tied = [11, 5, 33, 20]               # equal scores at the boundary
    b[hi] = np.arange(10, 10 + len(hi), dtype=np.float32)
    b[tied] = 5.0
    zero = torch.zeros((E, d), dtype=torch.int16, device="cuda")
    L = k.Layer(E, K, d, f, zero, pool.views, torch.from_numpy(b).cuda(), max_tokens=max(T, 1))
    L.set_option(k.K3MOE_OPT_MX, 1 if path == "mx" else 0)
    L.set_option(k.K3MOE_OPT_FUSED_T1, 1 if path == "fused" else 0)
    assert L.mx_t1() == (path == "mx")
    assert L.fused_t1() == (path == "fused")
    X = tokens_device(6, T, d, list(range(T)))
    out, ids, w = _run(L, X, T, K)
    rids, rw, _ = oracle.topk(np.zeros((T, E)), K, b.astype(np.float64))
    assert sorted(hi + [5, 11]) == list(rids[0])
    assert np.array_equal(ids, rids)
    assert np.allclose(w, 1.0 / K)  # the unbiased logits are all 0
    assert k.device_error() == 0
    L.close()


def test_degenerate_top_k(small):
    pool, Wr_bits, bias, E, K, d, f = small
    for kk in (1, 16):
        subs = margin_subs(5, 2, d, Wr_bits, kk)
        Xd = tokens(5, np.arange(2), d, subs)
        X = tokens_device(5, 2, d, subs)
        L = k.Layer(E, kk, d, f, router_tensor(Wr_bits), pool.views, max_tokens=2)
        for T in (1, 2):
            out, ids, w = _run(L, X[:T].contiguous(), T, kk)
            _check(pool, Wr_bits, None, kk, Xd[:T], out, ids, w)
        L.close()


def test_invalid_calls_are_refused(small):
    pool, Wr_bits, bias, E, K, d, f = small
    L = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, max_tokens=4)
    X = tokens_device(5, 4, d, [0] * 4)
    out = torch.empty((5, d), dtype=torch.float32, device="cuda")
    for T in (0, 5):
        with pytest.raises(k.K3Error) as ei:
            L.forward(X, T, out)
        assert ei.value.status == k.K3MOE_EINVAL
    L.close()
    with pytest.raises(k.K3Error):
        k.Layer(E, E + 1, d, f, router_tensor(Wr_bits), pool.views)


# ------------------------------------------------ full-size 896-expert layer

D, F, E896, K16 = 7168, 1536, 896, 16


@pytest.fixture(scope="module")
def full():
    pool = Pool(1, 0, E896, D, F)
    Wr_bits = synth.router_bf16(1, 0, E896, D)
    Wr = router_tensor(Wr_bits)
    bias = synth.bias_normal(1, 0, E896)
    L = k.Layer(E896, K16, D, F, Wr, pool.views, max_tokens=4096)
    Lb = k.Layer(E896, K16, D, F, Wr, pool.views, torch.from_numpy(bias).cuda(), max_tokens=4096)
    yield pool, Wr_bits, bias, L, Lb
    L.close()
    Lb.close()


def test_full_decode_batch1(full):
    """896 experts resident, x fp32, top-16, batch 1 (several tokens)."""
    pool, Wr_bits, bias, L, Lb = full
    T = 4
    subs = margin_subs(1, T, D, Wr_bits, K16)
    Xd = tokens(1, np.arange(T), D, subs)
    X = tokens_device(1, T, D, subs)
    for t in range(T):
        out, ids, w = _run(L, X[t:t + 1].contiguous(), 1, K16)
        _check(pool, Wr_bits, None, K16, Xd[t:t + 1], out, ids, w)


def test_full_batched_decode_64(full):
    """64 fp32 tokens grouped by expert; ids, weights and every output vector."""
    pool, Wr_bits, bias, L, Lb = full
    T = 64
    subs = margin_subs(1, T, D, Wr_bits, K16)
    Xd = tokens(1, np.arange(T), D, subs)
    X = tokens_device(1, T, D, subs)
    out, ids, w = _run(L, X, T, K16)
    _check(pool, Wr_bits, None, K16, Xd, out, ids, w, name="decode T=64")


def test_full_prefill_4096_bf16_biased(full):
    """4096 bf16 tokens with a per-expert selection bias ~ N(0,1); ids,
    weights and all 4096 output vectors (the heavily loaded experts span
    many tiles, so every tile edge and every scatter of the combine is
    seen)."""
    pool, Wr_bits, bias, L, Lb = full
    T = 4096
    subs = margin_subs(1, T, D, Wr_bits, K16, bias, bf16=True)
    Xd = tokens(1, np.arange(T), D, subs, bf16=True)
    X = tokens_device(1, T, D, subs, bf16=True)
    out, ids, w = _run(Lb, X, T, K16)
    counts = np.bincount(ids.ravel(), minlength=E896)
    assert counts.max() > 3 * counts.mean()  # the bias makes loads uneven
    _check(pool, Wr_bits, bias, K16, Xd, out, ids, w, name="prefill T=4096")


# ------------------------------------------- fused batch-1 kernel vs oracle

@pytest.fixture(scope="module")
def fusable():
    E, d, f = 48, 1024, 512
    pool = Pool(6, 0, E, d, f)
    Wr_bits = synth.router_bf16(6, 0, E, d)
    bias = synth.bias_normal(6, 0, E)
    return pool, Wr_bits, bias, E, d, f


@pytest.mark.parametrize("K,use_bias,act16", [(1, False, False), (8, True, False), (16, False, False),
                                              (16, True, True)])
def test_fused_batch1_matches_oracle_and_unfused(fusable, K, use_bias, act16):
    pool, Wr_bits, bias, E, d, f = fusable
    b = bias if use_bias else None
    bt = None if b is None else torch.from_numpy(b).cuda()
    T = 3
    subs = margin_subs(6, T, d, Wr_bits, K, b)
    Xd = tokens(6, np.arange(T), d, subs)
    X = tokens_device(6, T, d, subs)
    L = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, bt, max_tokens=1)
    L.set_option(k.K3MOE_OPT_MX, 0)
    assert L.fused_t1()
    if act16:
        L.set_option(k.K3MOE_OPT_ACT_F16, 1)
    L2 = k.Layer(E, K, d, f, router_tensor(Wr_bits), pool.views, bt, max_tokens=1)
    L2.set_option(k.K3MOE_OPT_MX, 0)
    L2.set_option(k.K3MOE_OPT_FUSED_T1, 0)
    assert not L2.fused_t1() and not L2.mx_t1()
    for t in range(T):
        out, ids, w = _run(L, X[t:t + 1].contiguous(), 1, K)
        _check(pool, Wr_bits, b, K, Xd[t:t + 1], out, ids, w)
        out2, ids2, w2 = _run(L2, X[t:t + 1].contiguous(), 1, K)
        assert np.array_equal(ids, ids2)
        # f16 activations: relative rounding 2^-12 per activation
        assert rel_err(out, out2) <= (1e-3 if act16 else 1e-5)
    # repeated launches reuse the grid-barrier counters
    for _ in range(5):
        out_again, _, _ = _run(L, X[0:1].contiguous(), 1, K)
    out0, _, _ = _run(L, X[0:1].contiguous(), 1, K)
    assert np.array_equal(out_again, out0)
    assert k.device_error() == 0
    L.close()
    L2.close()


@pytest.mark.parametrize("path", ["fused", "unfused"])
def test_full_decode_batch1_cuda_core_paths(full, path):
    """The two CUDA-core batch-1 paths on the full layer (the default there is
    the block-scaled tensor-core path, covered by test_full_decode_batch1)."""
    pool, Wr_bits, bias, L, Lb = full
    assert L.mx_t1()
    T = 2
    subs = margin_subs(1, T, D, Wr_bits, K16)
    Xd = tokens(1, np.arange(T), D, subs)
    X = tokens_device(1, T, D, subs)
    L.set_option(k.K3MOE_OPT_MX, 0)
    L.set_option(k.K3MOE_OPT_FUSED_T1, 1 if path == "fused" else 0)
    try:
        assert L.fused_t1() == (path == "fused")
        for t in range(T):
            out, ids, w = _run(L, X[t:t + 1].contiguous(), 1, K16)
            _check(pool, Wr_bits, None, K16, Xd[t:t + 1], out, ids, w)
    finally:
        L.set_option(k.K3MOE_OPT_FUSED_T1, 1)
        L.set_option(k.K3MOE_OPT_MX, 1)


def test_full_decode_batch1_f16_activations(full):
    """The opt-in f16-activation mode on the full layer stays inside the
    2e-3 bound; the measured error is printed for the record."""
    pool, Wr_bits, bias, L, Lb = full
    T = 3
    subs = margin_subs(1, T, D, Wr_bits, K16)
    Xd = tokens(1, np.arange(T), D, subs)
    X = tokens_device(1, T, D, subs)
    L.set_option(k.K3MOE_OPT_ACT_F16, 1)
    L.set_option(k.K3MOE_OPT_MX, 0)
    try:
        assert L.fused_t1()
        errs = []
        for t in range(T):
            out, ids, w = _run(L, X[t:t + 1].contiguous(), 1, K16)
            _check(pool, Wr_bits, None, K16, Xd[t:t + 1], out, ids, w)
            lg = oracle.router_logits(Xd[t:t + 1], Wr_bits)
            rids, rw, _ = oracle.topk(lg, K16)
            ref = oracle.combine(Xd[t:t + 1], rids, rw, pool.experts(rids[0]), pool.E)[0]
            errs.append(rel_err(out[0], ref))
        print("f16-activation max rel err per token:", ["%.2e" % e for e in errs])
    finally:
        L.set_option(k.K3MOE_OPT_ACT_F16, 0)
        L.set_option(k.K3MOE_OPT_MX, 1)
