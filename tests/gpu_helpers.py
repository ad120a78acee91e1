"""Shared helpers of the GPU parity tests: device upload of synthetic expert
pools, margin-checked tokens, and the error metric.  Inputs come only from
`synth`; expected values only from `oracle`."""
import numpy as np
import torch

import oracle
import synth
from mxfp4_routed_expert_select_gb300 import k3moe as k

TOL = 2e-3  # max_i |y_i - r_i| / max_i |r_i| per token (fp32 accumulation)


def rel_err(got, ref):
    """Normwise error of one token (the gate): max_i |y_i - r_i| / max_i |r_i|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-300))


def elem_err(got, ref):
    """Per-element relative error of one token, each denominator floored at
    1e-2 * max_i |r_i| (elements near zero would make the plain ratio
    meaningless): max_i |y_i - r_i| / max(|r_i|, 1e-2 max|r|).  Reported
    beside the normwise gate."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = max(1e-2 * np.max(np.abs(ref)), 1e-300)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


def batch_errors(got, ref):
    """(normwise, per-element) errors of every row of a [T, d] batch."""
    got = np.atleast_2d(got)
    ref = np.atleast_2d(ref)
    return (np.array([rel_err(g, r) for g, r in zip(got, ref)]),
            np.array([elem_err(g, r) for g, r in zip(got, ref)]))


def report(name, norm, elem):
    """One line of the errors a parity test measured (pytest -s shows it)."""
    print("%s: %d tokens, normwise max %.3e median %.3e; per-element (floor 1e-2 max|r|) "
          "max %.3e median %.3e" % (name, len(norm), np.max(norm), np.median(norm),
                                     np.max(elem), np.median(elem)))


class Pool:
    """E experts of one (pool, layer) in one device tensor of blobs."""

    def __init__(self, pool, layer, E, d, f, dev="cuda", e_lo=120, e_hi=130):
        self.pool, self.layer, self.E, self.d, self.f = pool, layer, E, d, f
        self.e_lo, self.e_hi = e_lo, e_hi
        self._cache = {}
        self.override = {}
        self.eb = k.expert_bytes(d, f)
        self.blobs = torch.empty((E, self.eb), dtype=torch.uint8, device=dev)
        for e in range(E):
            k.pack_expert(self.blobs[e], self.planes(e), d, f)
            if e % 64 == 63:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        self.views = [k.expert_view(self.blobs[e].data_ptr(), d, f) for e in range(E)]

    def planes(self, e):
        """Host planes of expert e (a test may replace an expert's planes by
        putting them in `override` after packing them onto the device)."""
        if e in self.override:
            return self.override[e]
        return synth.expert(self.pool, self.layer, e, self.d, self.f, self.e_lo, self.e_hi)

    def experts(self, ids):
        """Host planes of the given expert ids, for the oracle."""
        out = {}
        for e in set(int(v) for v in np.ravel(ids)):
            if e not in self._cache:
                if len(self._cache) > 96:
                    self._cache.clear()
                self._cache[e] = self.planes(e)
            out[e] = self._cache[e]
        return out


def router_tensor(bits, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev)


def margin_subs(pool, T, d, Wr_bits, k_, bias=None, gap=1e-3, bf16=False, max_tries=50,
                router="softmax"):
    """Per-token substream indices such that the oracle's rank-k / rank-k+1
    gap (on the router's selection key: logit + bias, or sigmoid(logit) +
    bias) is at least `gap`."""
    subs = np.zeros(T, np.int64)
    todo = np.arange(T)
    b = None if bias is None else np.asarray(bias, np.float64)
    for _ in range(max_tries):
        if todo.size == 0:
            return subs
        X = tokens(pool, todo, d, subs[todo], bf16)
        lg = oracle.router_logits(X, Wr_bits)
        _, _, m = oracle.topk(lg, k_, b, router)
        bad = m < gap
        subs[todo[bad]] += 1
        todo = todo[bad]
    raise RuntimeError("could not find margin tokens")


def tokens(pool, idx, d, subs, bf16=False):
    """fp64 copies of the activations (the values the GPU sees)."""
    rows = []
    for t, s in zip(np.ravel(idx), np.ravel(subs)):
        if bf16:
            b = synth.token_bf16(pool, int(t), d, int(s))
            rows.append((b.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
        else:
            rows.append(synth.token_f32(pool, int(t), d, int(s)).astype(np.float64))
    return np.stack(rows)


def tokens_device(pool, T, d, subs, bf16=False, dev="cuda"):
    if bf16:
        X = np.stack([synth.token_bf16(pool, t, d, int(subs[t])) for t in range(T)])
        return torch.from_numpy(X.view(np.int16)).to(dev).view(torch.bfloat16)
    X = np.stack([synth.token_f32(pool, t, d, int(subs[t])) for t in range(T)])
    return torch.from_numpy(X).to(dev)


# ------------------------------------------- MXFP4-activation path parity

MXQ_TAU = 3e-5  # reach of fp32 rounding, relative to a block's largest |h|
_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
_GAPS = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0])


def mxq_flip_bound(h32, Wd, wts):
    """Allowance (per output row) for the h codes whose rounding decision is
    within MXQ_TAU of the block maximum of a boundary: an element near an
    E2M1 midpoint may move one step (the gap at that midpoint); a block whose
    maximum is near a power of two may take the neighbouring scale, and its
    elements may then move by the difference between the two quantisations,
    both computed by the oracle's quantiser (the second on the block with its
    largest element moved just across the power of two).  h32 [n, f] fp32
    (the oracle's h rows of one expert), Wd [d, f] its dequantised down
    matrix, wts [n] the pairs' combine weights.
    Returns [n, d]: w * sum_i |Wd[r, i]| * delta_i."""
    n, f = h32.shape
    hb = np.abs(h32.astype(np.float64)).reshape(n, f // 32, 32)
    amax = hb.max(axis=2)
    _, E = np.frexp(amax)                       # amax = m 2^E, m in [0.5, 1)
    s = np.where(amax > 0, np.ldexp(1.0, E - 3), 1.0)  # 2^(floor(log2 amax) - 2)
    a = hb / s[..., None]
    tau_a = (MXQ_TAU * amax / s)[..., None]
    delta = np.zeros_like(hb)
    for m, g in zip(_MIDS, _GAPS):
        delta = np.maximum(delta, np.where(np.abs(a - m) <= tau_a, g, 0.0))
    delta *= s[..., None]
    p2 = np.exp2(np.round(np.log2(np.where(amax > 0, amax, 1.0))))
    near = (amax > 0) & (np.abs(amax / p2 - 1.0) <= MXQ_TAU)
    for r, b in zip(*np.nonzero(near)):
        blk = h32[r, 32 * b:32 * b + 32].astype(np.float32)
        i = int(np.argmax(np.abs(blk)))
        alt = blk.copy()
        # the largest element just across the power of two (same sign)
        alt[i] = np.float32(np.copysign(p2[r, b] * (1.0 - 2 * MXQ_TAU) if amax[r, b] >= p2[r, b]
                                        else p2[r, b], blk[i]))
        q0 = oracle.mx_quantize(blk)[0]
        q1 = oracle.mx_quantize(alt)[0]
        delta[r, b] = np.maximum(delta[r, b], np.abs(q1 - q0))
    delta = delta.reshape(n, f)
    return (delta @ np.abs(Wd).T) * np.asarray(wts, np.float64)[:, None]


def mxq_reference(Xd, rids, rw, planes_of):
    """(mode-B oracle output, flip allowance) for a batch."""
    T, d = Xd.shape
    bound = np.zeros((T, d))

    def acc(e, ts, js, h32, Wd):
        bound[ts] += mxq_flip_bound(h32, Wd, rw[ts, js])

    ref = oracle.combine_grouped_mxq(Xd, rids, rw, planes_of, on_expert=acc)
    return ref, bound


def mxq_check(out, ref, bound, name=None):
    """Gate: |out - ref| <= TOL * max|ref_t| + bound elementwise, per token.
    Returns (normwise errors, tokens with a non-zero allowance)."""
    out = np.asarray(out, np.float64)
    lim = TOL * np.max(np.abs(ref), axis=1, keepdims=True) + bound
    excess = np.abs(out - ref) - lim
    bad = np.nonzero(np.any(excess > 0, axis=1))[0]
    norm, elem = batch_errors(out, ref)
    if name:
        report(name + " vs mode-B oracle", norm, elem)
        print("%s: %d of %d tokens have a rounding-decision allowance (max %.3e of max|ref|)" %
              (name, int(np.count_nonzero(bound.max(axis=1) > 0)), len(out),
               float(np.max(bound.max(axis=1) / np.max(np.abs(ref), axis=1)))))
    assert bad.size == 0, [(int(t), float(norm[t])) for t in bad[:10]]
    return norm
