"""fp64 CPU oracle for the MXFP4 routed-expert MoE layer (ctypes front end).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product (the
CUDA library and its binding) never imports it and shares no code with it.

All arithmetic lives in ``k3oracle.c`` (plain C99, double precision); this
module only marshals numpy arrays.  Parity status per function is listed in
``k3oracle.c`` and in the tests under ``tests/test_oracle_*.py``.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3oracle.c")
_SO = os.path.join(_HERE, "libk3oracle.so")
_lib = None


def build(force=False):
    """Compile the oracle with gcc: plain C, fp64, contraction off."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class Mat(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("rows", ctypes.c_int), ("in_", ctypes.c_int)]


class Expert(ctypes.Structure):
    _fields_ = [("gate", Mat), ("up", Mat), ("down", Mat)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        p, i, d = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.orc_set_threads.argtypes = [i]
        L.orc_max_threads.restype = i
        L.orc_e2m1_value.restype = d
        L.orc_e2m1_value.argtypes = [i]
        L.orc_e8m0_value.restype = d
        L.orc_e8m0_value.argtypes = [i]
        L.orc_code.restype = i
        L.orc_code.argtypes = [p, i, i]
        L.orc_weight.restype = d
        L.orc_weight.argtypes = [p, i, i]
        L.orc_dequant.argtypes = [p, p]
        L.orc_matvec.argtypes = [p, p, p]
        L.orc_matvec_groupwise.argtypes = [p, p, p]
        L.orc_matrix_bytes.restype = ctypes.c_int64
        L.orc_matrix_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
        L.orc_expert_bytes.restype = ctypes.c_int64
        L.orc_expert_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
        L.orc_silu.restype = d
        L.orc_silu.argtypes = [d]
        L.orc_round_bf16.restype = d
        L.orc_round_bf16.argtypes = [d]
        L.orc_expert_forward_ex.argtypes = [p, p, p, i, p]
        L.orc_swiglu_n.argtypes = [p, p, ctypes.c_int64, i]
        L.orc_bf16_value.restype = d
        L.orc_bf16_value.argtypes = [ctypes.c_uint16]
        L.orc_router_logits.argtypes = [p, p, p, i, i, i]
        L.orc_topk_one.restype = d
        L.orc_topk.argtypes = [p, p, p, p, p, i, i, i]
        L.orc_topk_sigmoid.argtypes = [p, p, p, p, p, i, i, i, i]
        L.orc_mx_quant_block.restype = i
        L.orc_mx_quant_block.argtypes = [p, p]
        L.orc_mx_quantize.argtypes = [p, p, p, p, i]
        L.orc_expert_forward_mxq.argtypes = [p, p, p]
        L.orc_combine.argtypes = [p, p, i, i, p, p, i, p, i]
        L.orc_layer_forward.argtypes = [p, p, p, p, p, i, i, i, i, p, p, p, i]
        L.orc_rmsnorm.argtypes = [p, p, i, d]
        L.orc_shared_expert.argtypes = [p, p, p, p, p, i, i]
        L.orc_shared_forward.argtypes = [p, p, i, i, i, i, p, p, p]
        L.orc_cache_lru.restype = ctypes.c_longlong
        L.orc_cache_lru.argtypes = [p, p, p, i, i, p, i]
        L.orc_cache_belady.restype = ctypes.c_longlong
        L.orc_cache_belady.argtypes = [p, p, i, i]
        _lib = L
    return _lib


def set_threads(n):
    lib().orc_set_threads(int(n))


def max_threads():
    return lib().orc_max_threads()


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def make_mat(packed, scales):
    packed = _c(packed, np.uint8)
    scales = _c(scales, np.uint8)
    rows, half = packed.shape
    assert scales.shape == (rows, (2 * half) // 32)
    m = Mat(packed.ctypes.data, scales.ctypes.data, rows, 2 * half)
    m._keep = (packed, scales)
    return m


def make_expert(ex):
    """ctypes Expert from a dict with gate/up/down packed+scales planes."""
    g = make_mat(ex["gate_packed"], ex["gate_scales"])
    u = make_mat(ex["up_packed"], ex["up_scales"])
    dn = make_mat(ex["down_packed"], ex["down_scales"])
    e = Expert(g, u, dn)
    e._keep = (g, u, dn)
    return e


# ------------------------------------------------------------------ format

def e2m1_value(code):
    return lib().orc_e2m1_value(int(code))


def e8m0_value(e):
    return lib().orc_e8m0_value(int(e))


def code(packed, scales, r, j):
    m = make_mat(packed, scales)
    return lib().orc_code(ctypes.byref(m), r, j)


def dequant(packed, scales):
    m = make_mat(packed, scales)
    out = np.empty((m.rows, m.in_), np.float64)
    lib().orc_dequant(_p(out), ctypes.byref(m))
    return out


def matvec(packed, scales, x):
    m = make_mat(packed, scales)
    x = _c(x, np.float64)
    assert x.shape == (m.in_,)
    y = np.empty(m.rows, np.float64)
    lib().orc_matvec(_p(y), ctypes.byref(m), _p(x))
    return y


def matvec_groupwise(packed, scales, x):
    m = make_mat(packed, scales)
    x = _c(x, np.float64)
    y = np.empty(m.rows, np.float64)
    lib().orc_matvec_groupwise(_p(y), ctypes.byref(m), _p(x))
    return y


def matrix_bytes(rows, cols):
    return lib().orc_matrix_bytes(rows, cols)


def expert_bytes(d, f):
    return lib().orc_expert_bytes(d, f)


# ------------------------------------------------------------------ expert

def silu(z):
    return lib().orc_silu(float(z))


def round_bf16(v):
    return lib().orc_round_bf16(float(v))


def expert_forward(ex, x, h_bf16=False, want_h=False):
    e = make_expert(ex)
    x = _c(x, np.float64)
    d = e.gate.in_
    f = e.gate.rows
    assert x.shape == (d,)
    y = np.empty(d, np.float64)
    h = np.empty(f, np.float64) if want_h else None
    lib().orc_expert_forward_ex(_p(y), ctypes.byref(e), _p(x), int(bool(h_bf16)), _p(h))
    return (y, h) if want_h else y


def mx_quantize(x):
    """MXFP4 quantisation of fp32 activations (OCP rule): (values float64 [n],
    codes uint8 [n], scale bytes uint8 [n/32]); n a multiple of 32."""
    x = _c(x, np.float32).ravel()
    assert x.size % 32 == 0
    xq = np.empty(x.size, np.float64)
    codes = np.empty(x.size, np.uint8)
    sc = np.empty(x.size // 32, np.uint8)
    lib().orc_mx_quantize(_p(xq), _p(codes), _p(sc), _p(x), x.size)
    return xq, codes, sc


def expert_forward_mxq(ex, x):
    """One expert with MXFP4-quantised activations x (fp32 [d]) and h."""
    e = make_expert(ex)
    x = _c(x, np.float32)
    y = np.empty(e.gate.in_, np.float64)
    lib().orc_expert_forward_mxq(_p(y), ctypes.byref(e), _p(x))
    return y


# ------------------------------------------------------------------ router

def bf16_value(bits):
    return lib().orc_bf16_value(int(bits))


def router_logits(x, Wr_bits):
    x = _c(np.atleast_2d(x), np.float64)
    Wr = _c(Wr_bits, np.uint16)
    T, d = x.shape
    E = Wr.shape[0]
    assert Wr.shape == (E, d)
    out = np.empty((T, E), np.float64)
    lib().orc_router_logits(_p(out), _p(x), _p(Wr), T, E, d)
    return out


ROUTERS = ("softmax", "sigmoid", "sigmoid_norm")


def topk(logits, k, bias=None, router="softmax"):
    """(ids ascending int32 [T,k], weights [T,k], margins [T]).

    router "softmax": select on logit + bias, weights = softmax of the
    unbiased selected logits.  "sigmoid" / "sigmoid_norm": select on
    sigmoid(logit) + bias, weights = the unbiased sigmoid scores, as they are
    or renormalised over the chosen set."""
    logits = _c(np.atleast_2d(logits), np.float64)
    T, E = logits.shape
    b = None if bias is None else _c(bias, np.float64)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    m = np.empty(T, np.float64)
    if router == "softmax":
        lib().orc_topk(_p(ids), _p(w), _p(m), _p(logits), _p(b), T, E, k)
    elif router in ("sigmoid", "sigmoid_norm"):
        lib().orc_topk_sigmoid(_p(ids), _p(w), _p(m), _p(logits), _p(b), T, E, k,
                               1 if router == "sigmoid_norm" else 0)
    else:
        raise ValueError(router)
    return ids, w, m


def _expert_table(experts, E):
    """experts: dict id -> expert dict (only the ids that are read)."""
    tab = (Expert * E)()
    keep = []
    for e, ex in experts.items():
        ce = make_expert(ex)
        tab[e] = ce
        keep.append(ce)
    tab._keep = keep
    return tab


def combine(x, ids, w, experts, E, h_bf16=False):
    x = _c(np.atleast_2d(x), np.float64)
    T, d = x.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    k = ids.shape[1]
    need = set(int(v) for v in ids.ravel())
    assert need <= set(experts), "missing expert weights for ids %s" % sorted(need - set(experts))
    tab = _expert_table(experts, E)
    out = np.empty((T, d), np.float64)
    lib().orc_combine(_p(out), _p(x), T, d, _p(ids), _p(w), k,
                      ctypes.cast(tab, ctypes.c_void_p), int(bool(h_bf16)))
    return out


def combine_grouped(x, ids, w, planes_of, h_bf16=False):
    """The same weighted sum as ``combine``, grouped by expert: every selected
    expert's three matrices are dequantised once (``dequant``, the pinned
    definition) and applied to all of its tokens with a library matrix
    product in fp64; SwiGLU is ``orc_silu`` (and ``orc_round_bf16``) element
    by element.  ``planes_of(e)`` returns the expert's planes, so only one
    expert is held at a time.  It differs from ``combine`` only in the order
    of the fp64 sums (checked on the CPU), and makes whole-batch checks of
    thousands of tokens affordable."""
    x = _c(np.atleast_2d(x), np.float64)
    T, d = x.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    out = np.zeros((T, d), np.float64)
    for e in np.unique(ids):
        ts, js = np.nonzero(ids == e)
        ex = planes_of(int(e))
        Xe = x[ts]
        g = Xe @ dequant(ex["gate_packed"], ex["gate_scales"]).T
        u = Xe @ dequant(ex["up_packed"], ex["up_scales"]).T
        g = np.ascontiguousarray(g)
        u = np.ascontiguousarray(u)
        lib().orc_swiglu_n(_p(g), _p(u), g.size, int(bool(h_bf16)))
        y = g @ dequant(ex["down_packed"], ex["down_scales"]).T
        # a token selects an expert at most once, so ts has no repeats
        out[ts] += w[ts, js][:, None] * y
    return out


def combine_grouped_mxq(x, ids, w, planes_of, on_expert=None):
    """The layer with MXFP4-quantised activations, grouped by expert: the
    steps of ``expert_forward_mxq`` (x quantised per 32-block by
    ``mx_quantize``; g and u in fp64 from the dequantised weights; h =
    silu(g) u rounded to fp32 and quantised the same way; y = W_down h_q),
    each expert's tokens in one library matrix product, weighted and summed
    as in ``combine``.  ``on_expert(e, ts, js, h32, Wd)``, if given, sees
    every expert's fp32 h rows and its dequantised down matrix (for a
    test's tolerance of rounding decisions)."""
    x = _c(np.atleast_2d(x), np.float64)
    T, d = x.shape
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    xq = mx_quantize(x.astype(np.float32).ravel())[0].reshape(T, d)
    out = np.zeros((T, d), np.float64)
    for e in np.unique(ids):
        ts, js = np.nonzero(ids == e)
        ex = planes_of(int(e))
        Xe = xq[ts]
        g = np.ascontiguousarray(Xe @ dequant(ex["gate_packed"], ex["gate_scales"]).T)
        u = np.ascontiguousarray(Xe @ dequant(ex["up_packed"], ex["up_scales"]).T)
        lib().orc_swiglu_n(_p(g), _p(u), g.size, 0)
        h32 = g.astype(np.float32)
        hq = mx_quantize(h32.ravel())[0].reshape(h32.shape)
        Wd = dequant(ex["down_packed"], ex["down_scales"])
        y = hq @ Wd.T
        # a token selects an expert at most once, so ts has no repeats
        out[ts] += w[ts, js][:, None] * y
        if on_expert is not None:
            on_expert(int(e), ts, js, h32, Wd)
    return out


def layer_forward(x, Wr_bits, k, experts, bias=None, h_bf16=False):
    """Full layer. `experts` must hold (at least) every expert selected."""
    x = _c(np.atleast_2d(x), np.float64)
    T, d = x.shape
    E = Wr_bits.shape[0]
    logits = router_logits(x, Wr_bits)
    ids, w, m = topk(logits, k, bias)
    out = combine(x, ids, w, experts, E, h_bf16)
    return out, ids, w, m


def shared_expert(ex, x):
    """One bf16 shared expert: ex = dict(gate [f, d], up [f, d], down [d, f])
    as bf16 bit patterns (uint16); x [d].  Returns y [d] in fp64."""
    g = _c(ex["gate"], np.uint16)
    u = _c(ex["up"], np.uint16)
    dn = _c(ex["down"], np.uint16)
    f, d = g.shape
    assert u.shape == (f, d) and dn.shape == (d, f)
    x = _c(x, np.float64)
    assert x.shape == (d,)
    y = np.empty(d, np.float64)
    lib().orc_shared_expert(_p(y), _p(g), _p(u), _p(dn), _p(x), d, f)
    return y


def shared_forward(x, experts):
    """out[t] = sum_s shared_expert(experts[s], x[t]); x [T, d] fp64."""
    x = _c(np.atleast_2d(x), np.float64)
    T, d = x.shape
    arrs = [(_c(e["gate"], np.uint16), _c(e["up"], np.uint16), _c(e["down"], np.uint16)) for e in experts]
    f = arrs[0][0].shape[0]
    n = len(arrs)
    P = ctypes.c_void_p * n
    gates = P(*[a[0].ctypes.data for a in arrs])
    ups = P(*[a[1].ctypes.data for a in arrs])
    downs = P(*[a[2].ctypes.data for a in arrs])
    out = np.empty((T, d), np.float64)
    lib().orc_shared_forward(_p(out), _p(x), T, d, f, n, ctypes.cast(gates, ctypes.c_void_p),
                             ctypes.cast(ups, ctypes.c_void_p), ctypes.cast(downs, ctypes.c_void_p))
    return out


def rmsnorm(x, eps):
    x = _c(x, np.float64)
    y = np.empty_like(x)
    lib().orc_rmsnorm(_p(y), _p(x), x.size, float(eps))
    return y


# ------------------------------------------------------------------- cache

def cache_lru(keys, batch_len, capacity, pinned=()):
    keys = _c(keys, np.int64)
    bl = _c(batch_len, np.int32)
    pn = _c(np.asarray(pinned, np.int64), np.int64)
    hit = np.zeros(keys.size, np.uint8)
    h = lib().orc_cache_lru(_p(hit), _p(keys), _p(bl), bl.size, int(capacity),
                            _p(pn) if pn.size else None, pn.size)
    return h, hit


def cache_belady(keys, batch_len, capacity):
    keys = _c(keys, np.int64)
    bl = _c(batch_len, np.int32)
    return lib().orc_cache_belady(_p(keys), _p(bl), bl.size, int(capacity))
