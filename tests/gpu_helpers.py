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
