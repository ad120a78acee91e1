"""ctypes binding of libk3moe.so (the C ABI in include/k3moe.h).

Argument marshalling only: every step of the MoE layer runs in the library's
CUDA kernels.  Device memory and streams come from PyTorch; tensors are passed
as raw pointers.  Importing this module fails loudly when the compiled library
is missing -- there is no CPU fallback.
"""
import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
# K3MOE_LIBRARY may name another build of the same library (e.g. a debug build)
SO = os.environ.get("K3MOE_LIBRARY") or os.path.join(HERE, "libk3moe.so")

K3MOE_OK = 0
K3MOE_EINVAL = -1
K3MOE_ENOMEM = -2
K3MOE_ECUDA = -3
K3MOE_ETIMEOUT = -4
K3MOE_EBUSY = -5
K3MOE_ENODEV = -6
K3MOE_EIO = -7
K3MOE_POLICY_LRU = 0
K3MOE_POLICY_BELADY = 1
K3MOE_F32 = 0
K3MOE_BF16 = 1
K3MOE_OPT_FUSED_T1 = 1
K3MOE_OPT_ACT_F16 = 2
K3MOE_OPT_TC = 4
K3MOE_OPT_TC_E4M3 = 8
K3MOE_OPT_MX = 16
K3MOE_OPT_SIGMOID_ROUTER = 32
K3MOE_OPT_SIGMOID_NORM = 64
K3MOE_OPT_MXQ = 128
K3MOE_NOALLOC_MAX_F = 2048


class K3Error(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s failed: %s (%d)" % (what, strerror(status), status))
        self.status = status


class Mat(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("rows", ctypes.c_int32), ("in_", ctypes.c_int32)]


class Expert(ctypes.Structure):
    _fields_ = [("gate", Mat), ("up", Mat), ("down", Mat)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("router_w", ctypes.c_void_p), ("sel_bias", ctypes.c_void_p),
                ("host_experts", ctypes.c_void_p), ("max_tokens", ctypes.c_int32)]


class CacheStats(ctypes.Structure):
    _fields_ = [("lookups", ctypes.c_int64), ("hits", ctypes.c_int64),
                ("misses", ctypes.c_int64), ("evictions", ctypes.c_int64),
                ("h2d_bytes", ctypes.c_int64), ("hbm_bytes", ctypes.c_int64),
                ("slots", ctypes.c_int32), ("pinned", ctypes.c_int32),
                ("inflight", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class TrunkStats(ctypes.Structure):
    _fields_ = [("requests", ctypes.c_int64), ("resident", ctypes.c_int64),
                ("prefetched", ctypes.c_int64), ("h2d_bytes", ctypes.c_int64),
                ("n_layers", ctypes.c_int32), ("pinned_layers", ctypes.c_int32),
                ("ring_slots", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class StreamDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("host_layers", ctypes.c_void_p),
                ("cache", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("trunk", ctypes.c_void_p), ("n_shared", ctypes.c_int32)]


class Bf16Expert(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p)]


ALLOC_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                            ctypes.POINTER(ctypes.c_void_p))
FREE_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p)
COPY_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_size_t)
SLOT_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int32)


class Copier(ctypes.Structure):
    _fields_ = [("ctx", ctypes.c_void_p), ("alloc_arena", ALLOC_FN), ("free_arena", FREE_FN),
                ("copy", COPY_FN), ("wait", SLOT_FN), ("release", SLOT_FN)]


# Every exported symbol with its (restype, argtypes).
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "k3moe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "k3moe_version": (ctypes.c_int, []),
    "k3moe_device_error": (ctypes.c_int, []),
    "k3moe_check_wait_timeout": (ctypes.c_int, [ctypes.c_void_p]),
    "k3moe_matrix_bytes": (_I64, [_I, _I]),
    "k3moe_expert_bytes": (_I64, [_I, _I]),
    "k3moe_expert_view": (ctypes.c_int, [_P, _P, _I, _I]),
    "k3moe_pack_expert": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "k3moe_matmul_mxfp4": (ctypes.c_int, [_P, _P, _P, _P]),
    "k3moe_expert_gemv_workspace": (_SZ, [_I, _I]),
    "k3moe_expert_gemv": (ctypes.c_int, [_P, _P, _P, _I, _I, _P, _SZ, _P]),
    "k3moe_expert_gemv_noalloc": (ctypes.c_int, [_P, _P, _P, _I, _I, _P]),
    "k3moe_layer_create": (ctypes.c_int, [_P, _P]),
    "k3moe_layer_destroy": (ctypes.c_int, [_P]),
    "k3moe_layer_route": (ctypes.c_int, [_P, _P, ctypes.c_int, _I, _P, _P, _P]),
    "k3moe_layer_forward": (ctypes.c_int, [_P, _P, ctypes.c_int, _I, _P, _P, _P, _P]),
    "k3moe_layer_experts_t1": (ctypes.c_int, [_P, _P, _P, _P, _I, _P, _P]),
    "k3moe_layer_set_events": (ctypes.c_int, [_P, _P, _I]),
    "k3moe_layer_set_option": (ctypes.c_int, [_P, _I, _I]),
    "k3moe_layer_fused_t1": (ctypes.c_int, [_P]),
    "k3moe_layer_mx_t1": (ctypes.c_int, [_P]),
    "k3moe_layer_mxq": (ctypes.c_int, [_P]),
    "k3moe_shared_expert_bytes": (_I64, [_I, _I]),
    "k3moe_shared_expert_view": (ctypes.c_int, [_P, _P, _I, _I]),
    "k3moe_shared_workspace": (_SZ, [_I, _I]),
    "k3moe_shared_forward": (ctypes.c_int, [_P, _P, _I, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "k3moe_mx_quantize": (ctypes.c_int, [_P, _P, _P, _I, _I, _I, _P]),
    "k3moe_rmsnorm": (ctypes.c_int, [_P, _P, _I, _F, _P]),
    "k3moe_residual_add": (ctypes.c_int, [_P, _P, _I, _P]),
    "k3moe_cache_create": (ctypes.c_int, [_P, _SZ, _SZ, _P, _I, _I]),
    "k3moe_cache_destroy": (ctypes.c_int, [_P]),
    "k3moe_cache_acquire": (ctypes.c_int, [_P, _P, _I, _P, _P, _P]),
    "k3moe_cache_acquire_split": (ctypes.c_int, [_P, _P, _I, _P, _P, _P]),
    "k3moe_cache_wait_copies": (ctypes.c_int, [_P, _P]),
    "k3moe_cache_wait_copy": (ctypes.c_int, [_P, _P, _P]),
    "k3moe_cache_release": (ctypes.c_int, [_P, _P]),
    "k3moe_cache_pin": (ctypes.c_int, [_P, _I64, _P]),
    "k3moe_cache_get_stats": (ctypes.c_int, [_P, _P]),
    "k3moe_cache_histogram": (ctypes.POINTER(ctypes.c_uint32), [_P]),
    "k3moe_cache_create_with_copier": (ctypes.c_int, [_P, _SZ, _SZ, _P, _I, _I, _P]),
    "k3moe_cache_slot_of": (_I, [_P, _I64]),
    "k3moe_cache_trace_record": (ctypes.c_int, [_P, _I]),
    "k3moe_cache_trace_get": (ctypes.c_int, [_P, _P, _I64, _P, _I, _P, _P]),
    "k3moe_cache_pin_hot": (ctypes.c_int, [_P, _I, _P]),
    "k3moe_cache_unpin": (ctypes.c_int, [_P, _I64]),
    "k3moe_trace_replay": (ctypes.c_int, [_P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "k3moe_trace_sweep": (ctypes.c_int, [_P, _P, _I, _P, _I, _I, _P]),
    "k3moe_trace_pin_sweep": (ctypes.c_int, [_P, _P, _I, _I, _P, _P, _I, _I64, _P]),
    "k3moe_hot_set": (ctypes.c_int, [_P, _I64, _I, _P]),
    "k3moe_trace_save": (ctypes.c_int, [ctypes.c_char_p, _P, _P, _I]),
    "k3moe_trace_load": (ctypes.c_int, [ctypes.c_char_p, _P, _I64, _P, _I, _P, _P]),
    "k3moe_stream_decode": (ctypes.c_int, [_P, _P, _I, _P, _P, _P, _P]),
    "k3moe_trunk_create": (ctypes.c_int, [_P, _P, _P, _I, _SZ, _I]),
    "k3moe_trunk_create_with_copier": (ctypes.c_int, [_P, _P, _P, _I, _SZ, _I, _P]),
    "k3moe_trunk_destroy": (ctypes.c_int, [_P]),
    "k3moe_trunk_acquire": (ctypes.c_int, [_P, _I, _P, _P, _P]),
    "k3moe_trunk_release": (ctypes.c_int, [_P, _I, _P]),
    "k3moe_trunk_get_stats": (ctypes.c_int, [_P, _P]),
}

_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            raise ImportError("libk3moe.so is not built (run __graft_entry__.build()); "
                              "there is no CPU fallback")
        L = ctypes.CDLL(SO)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def strerror(st):
    return lib().k3moe_strerror(st).decode()


def check(st, what):
    if st != K3MOE_OK:
        raise K3Error(st, what)
    return st


# --------------------------------------------------------------- helpers

def _ptr(t):
    """Raw pointer of a torch tensor / numpy array / int / None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(s=None):
    import torch
    if s is None:
        s = torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else s


def matrix_bytes(rows, cols):
    return lib().k3moe_matrix_bytes(rows, cols)


def expert_bytes(d, f):
    return lib().k3moe_expert_bytes(d, f)


def expert_view(blob_ptr, d, f):
    e = Expert()
    check(lib().k3moe_expert_view(ctypes.byref(e), blob_ptr, d, f), "k3moe_expert_view")
    return e


def host_plane_views(blob_ptr, d, f):
    """numpy views of the six planes inside a HOST blob (for filling it)."""
    e = expert_view(blob_ptr, d, f)

    def arr(p, rows, cols):
        buf = (ctypes.c_uint8 * (rows * cols)).from_address(p)
        return np.frombuffer(buf, np.uint8).reshape(rows, cols)
    return dict(gate_packed=arr(e.gate.packed, f, d // 2), gate_scales=arr(e.gate.scales, f, d // 32),
                up_packed=arr(e.up.packed, f, d // 2), up_scales=arr(e.up.scales, f, d // 32),
                down_packed=arr(e.down.packed, d, f // 2), down_scales=arr(e.down.scales, d, f // 32))


def pack_expert(blob, planes, d, f, stream=None):
    """Copy the six canonical planes (numpy or tensors) into a device blob."""
    ps = [planes[k] for k in ("gate_packed", "gate_scales", "up_packed", "up_scales",
                              "down_packed", "down_scales")]
    ps = [np.ascontiguousarray(p) if isinstance(p, np.ndarray) else p for p in ps]
    check(lib().k3moe_pack_expert(_ptr(blob), *[_ptr(p) for p in ps], d, f, _stream(stream)),
          "k3moe_pack_expert")
    return ps  # keep host arrays alive until the copies are done


def matmul_mxfp4(y, x, packed, scales, rows, cols, stream=None):
    m = Mat(_ptr(packed), _ptr(scales), rows, cols)
    check(lib().k3moe_matmul_mxfp4(_ptr(y), _ptr(x), ctypes.byref(m), _stream(stream)),
          "k3moe_matmul_mxfp4")


def expert_gemv_workspace(d, f):
    return lib().k3moe_expert_gemv_workspace(d, f)


def expert_gemv(y, x, expert, d, f, workspace, stream=None):
    nbytes = workspace.numel() * workspace.element_size()
    check(lib().k3moe_expert_gemv(_ptr(y), _ptr(x), ctypes.byref(expert), d, f, _ptr(workspace),
                                  nbytes, _stream(stream)), "k3moe_expert_gemv")


def mx_quantize(codes, scales, x, rows, cols, stream=None):
    """MXFP4 quantisation of activations (k3moe_mx_quantize): x [rows][cols]
    (fp32 or bf16 tensor) -> codes uint8 [rows][cols/2], scales uint8
    [rows][cols/32]."""
    import torch
    dt = K3MOE_BF16 if x.dtype == torch.bfloat16 else K3MOE_F32
    check(lib().k3moe_mx_quantize(_ptr(codes), _ptr(scales), _ptr(x), dt, rows, cols, _stream(stream)),
          "k3moe_mx_quantize")


def expert_gemv_noalloc(y, x, expert, d, f, stream=None):
    """k3moe_expert_gemv without a workspace (static device scratch)."""
    check(lib().k3moe_expert_gemv_noalloc(_ptr(y), _ptr(x), ctypes.byref(expert), d, f,
                                          _stream(stream)), "k3moe_expert_gemv_noalloc")


def rmsnorm(u, x, eps, stream=None):
    check(lib().k3moe_rmsnorm(_ptr(u), _ptr(x), x.numel(), eps, _stream(stream)), "k3moe_rmsnorm")


def residual_add(x, delta, stream=None):
    check(lib().k3moe_residual_add(_ptr(x), _ptr(delta), x.numel(), _stream(stream)),
          "k3moe_residual_add")


def device_error():
    return lib().k3moe_device_error()


class Layer:
    """k3moe_layer_* : router, top-k and the expert products of one layer."""

    def __init__(self, n_experts, top_k, d, f, router_w, expert_views, sel_bias=None,
                 max_tokens=1):
        self.E, self.k, self.d, self.f = n_experts, top_k, d, f
        if expert_views is None:
            self._views = None
            views_ptr = None
        else:
            self._views = (Expert * n_experts)(*expert_views)
            views_ptr = ctypes.cast(self._views, ctypes.c_void_p)
        desc = LayerDesc(n_experts, top_k, d, f, _ptr(router_w), _ptr(sel_bias), views_ptr,
                         max_tokens)
        h = ctypes.c_void_p()
        check(lib().k3moe_layer_create(ctypes.byref(h), ctypes.byref(desc)), "k3moe_layer_create")
        self.h = h
        self._keep = (router_w, sel_bias)

    def forward(self, X, T, out, ids_out=None, w_out=None, stream=None):
        import torch
        dt = K3MOE_BF16 if X.dtype == torch.bfloat16 else K3MOE_F32
        check(lib().k3moe_layer_forward(self.h, _ptr(X), dt, T, _ptr(out), _ptr(ids_out),
                                        _ptr(w_out), _stream(stream)), "k3moe_layer_forward")

    def route(self, X, T, ids, w, stream=None):
        import torch
        dt = K3MOE_BF16 if X.dtype == torch.bfloat16 else K3MOE_F32
        check(lib().k3moe_layer_route(self.h, _ptr(X), dt, T, _ptr(ids), _ptr(w), _stream(stream)),
              "k3moe_layer_route")

    def set_option(self, option, value):
        check(lib().k3moe_layer_set_option(self.h, option, int(value)), "k3moe_layer_set_option")

    def fused_t1(self):
        return lib().k3moe_layer_fused_t1(self.h) == 1

    def mx_t1(self):
        return lib().k3moe_layer_mx_t1(self.h) == 1

    def mxq(self):
        return lib().k3moe_layer_mxq(self.h) == 1

    def set_events(self, events):
        """events: 4 torch.cuda.Event (or None to clear); each must have been
        recorded once (torch creates the CUDA event lazily)."""
        if not events:
            check(lib().k3moe_layer_set_events(self.h, None, 0), "k3moe_layer_set_events")
            return
        arr = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        check(lib().k3moe_layer_set_events(self.h, ctypes.cast(arr, ctypes.c_void_p), 4),
              "k3moe_layer_set_events")

    def experts_t1(self, x, sel_views, w, out, stream=None):
        arr = (Expert * len(sel_views))(*sel_views)
        check(lib().k3moe_layer_experts_t1(self.h, _ptr(x), ctypes.cast(arr, ctypes.c_void_p),
                                           _ptr(w), len(sel_views), _ptr(out), _stream(stream)),
              "k3moe_layer_experts_t1")

    def close(self):
        if self.h:
            lib().k3moe_layer_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Cache:
    """k3moe_cache_* : HBM LRU expert cache over host blobs."""

    def __init__(self, capacity_bytes, expert_bytes_, host_blob_ptrs, n_layers, n_experts,
                 copier=None):
        n = n_layers * n_experts
        self._blobs = (ctypes.c_void_p * n)(*host_blob_ptrs)
        h = ctypes.c_void_p()
        if copier is None:
            st = lib().k3moe_cache_create(ctypes.byref(h), capacity_bytes, expert_bytes_,
                                          ctypes.cast(self._blobs, ctypes.c_void_p), n_layers,
                                          n_experts)
        else:
            self._copier = copier
            st = lib().k3moe_cache_create_with_copier(ctypes.byref(h), capacity_bytes,
                                                      expert_bytes_,
                                                      ctypes.cast(self._blobs, ctypes.c_void_p),
                                                      n_layers, n_experts, ctypes.byref(copier))
        check(st, "k3moe_cache_create")
        self.h = h
        self.nkeys = n

    def acquire(self, keys, stream=0, raise_on_error=True, split=False):
        """split=True: k3moe_cache_acquire_split (misses usable only after
        wait_copies)."""
        keys = np.ascontiguousarray(keys, np.int64)
        n = keys.size
        out = (ctypes.c_void_p * n)()
        hit = np.zeros(n, np.uint8)
        name = "k3moe_cache_acquire_split" if split else "k3moe_cache_acquire"
        st = getattr(lib(), name)(self.h, keys.ctypes.data, n,
                                  ctypes.cast(out, ctypes.c_void_p), hit.ctypes.data, stream)
        if raise_on_error:
            check(st, name)
        return [out[i] for i in range(n)], hit, st

    def wait_copies(self, stream=0):
        return lib().k3moe_cache_wait_copies(self.h, stream)

    def wait_copy(self, blob_ptr, stream=0):
        return lib().k3moe_cache_wait_copy(self.h, blob_ptr, stream)

    def release(self, stream=0):
        return check(lib().k3moe_cache_release(self.h, stream), "k3moe_cache_release")

    def pin(self, key, stream=0):
        return lib().k3moe_cache_pin(self.h, int(key), stream)

    def stats(self):
        s = CacheStats()
        check(lib().k3moe_cache_get_stats(self.h, ctypes.byref(s)), "k3moe_cache_get_stats")
        return s.as_dict()

    def histogram(self):
        p = lib().k3moe_cache_histogram(self.h)
        return np.ctypeslib.as_array(p, shape=(self.nkeys,)).copy()

    def slot_of(self, key):
        return lib().k3moe_cache_slot_of(self.h, int(key))

    def record_trace(self, on=True):
        """k3moe_cache_trace_record: start (clearing the record) or stop."""
        check(lib().k3moe_cache_trace_record(self.h, 1 if on else 0), "k3moe_cache_trace_record")

    def trace(self):
        """k3moe_cache_trace_get: (keys int64, batch_len int32) recorded so far."""
        nk, nb = ctypes.c_int64(), ctypes.c_int32()
        check(lib().k3moe_cache_trace_get(self.h, None, 0, None, 0, ctypes.byref(nk),
                                          ctypes.byref(nb)), "k3moe_cache_trace_get")
        keys = np.zeros(nk.value, np.int64)
        bl = np.zeros(nb.value, np.int32)
        check(lib().k3moe_cache_trace_get(self.h, keys.ctypes.data, keys.size, bl.ctypes.data,
                                          bl.size, ctypes.byref(nk), ctypes.byref(nb)),
              "k3moe_cache_trace_get")
        return keys, bl

    def pin_hot(self, n, stream=0):
        """k3moe_cache_pin_hot: pin the n most requested keys."""
        return lib().k3moe_cache_pin_hot(self.h, int(n), stream)

    def unpin(self, key):
        return check(lib().k3moe_cache_unpin(self.h, int(key)), "k3moe_cache_unpin")

    def close(self):
        if self.h:
            lib().k3moe_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Trunk:
    """k3moe_trunk_* : per-layer weights as a resident prefix plus a ring of
    streaming slots."""

    def __init__(self, host_layer_ptrs, layer_bytes, pinned_bytes, ring_slots, copier=None):
        n = len(host_layer_ptrs)
        self._ptrs = (ctypes.c_void_p * n)(*host_layer_ptrs)
        self._bytes = (ctypes.c_size_t * n)(*layer_bytes)
        h = ctypes.c_void_p()
        if copier is None:
            st = lib().k3moe_trunk_create(ctypes.byref(h), ctypes.cast(self._ptrs, ctypes.c_void_p),
                                          ctypes.cast(self._bytes, ctypes.c_void_p), n,
                                          int(pinned_bytes), int(ring_slots))
        else:
            self._copier = copier
            st = lib().k3moe_trunk_create_with_copier(
                ctypes.byref(h), ctypes.cast(self._ptrs, ctypes.c_void_p),
                ctypes.cast(self._bytes, ctypes.c_void_p), n, int(pinned_bytes), int(ring_slots),
                ctypes.byref(copier))
        check(st, "k3moe_trunk_create")
        self.h = h

    def acquire(self, layer, stream=0, raise_on_error=True):
        """(device pointer, resident flag, status)."""
        p = ctypes.c_void_p()
        res = ctypes.c_uint8()
        st = lib().k3moe_trunk_acquire(self.h, int(layer), ctypes.byref(p), ctypes.byref(res), stream)
        if raise_on_error:
            check(st, "k3moe_trunk_acquire")
        return p.value, res.value, st

    def release(self, layer, stream=0):
        return lib().k3moe_trunk_release(self.h, int(layer), stream)

    def stats(self):
        s = TrunkStats()
        check(lib().k3moe_trunk_get_stats(self.h, ctypes.byref(s)), "k3moe_trunk_get_stats")
        return s.as_dict()

    def close(self):
        if self.h:
            lib().k3moe_trunk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_POLICIES = {"lru": K3MOE_POLICY_LRU, "belady": K3MOE_POLICY_BELADY}


def _trace_arrays(keys, batch_len):
    return np.ascontiguousarray(keys, np.int64), np.ascontiguousarray(batch_len, np.int32)


def trace_replay(keys, batch_len, capacity, policy="lru", pinned=()):
    """k3moe_trace_replay: (hit count, uint8 hit flag per key); the status
    K3MOE_EBUSY is returned as a hit count of -1."""
    keys, bl = _trace_arrays(keys, batch_len)
    pin = np.ascontiguousarray(pinned, np.int64)
    hit = np.zeros(keys.size, np.uint8)
    hits = ctypes.c_int64(-1)
    st = lib().k3moe_trace_replay(keys.ctypes.data, bl.ctypes.data, bl.size, int(capacity),
                                  _POLICIES[policy], pin.ctypes.data if pin.size else None,
                                  pin.size, hit.ctypes.data, ctypes.byref(hits))
    if st == K3MOE_EBUSY:
        return -1, hit
    check(st, "k3moe_trace_replay")
    return hits.value, hit


def trace_sweep(keys, batch_len, capacities, policy="lru"):
    """k3moe_trace_sweep: hit counts per capacity (-1 where a batch does not fit)."""
    keys, bl = _trace_arrays(keys, batch_len)
    caps = np.ascontiguousarray(capacities, np.int32)
    out = np.zeros(caps.size, np.int64)
    check(lib().k3moe_trace_sweep(keys.ctypes.data, bl.ctypes.data, bl.size, caps.ctypes.data,
                                  caps.size, _POLICIES[policy], out.ctypes.data),
          "k3moe_trace_sweep")
    return out


def trace_pin_sweep(keys, batch_len, capacity, hot_keys, pin_counts, count_from=0):
    """k3moe_trace_pin_sweep: LRU hits at positions >= count_from with the
    first pin_counts[c] hot keys pinned, per c (-1 where a batch does not fit)."""
    keys, bl = _trace_arrays(keys, batch_len)
    hot = np.ascontiguousarray(hot_keys, np.int64)
    pc = np.ascontiguousarray(pin_counts, np.int32)
    out = np.zeros(pc.size, np.int64)
    check(lib().k3moe_trace_pin_sweep(keys.ctypes.data, bl.ctypes.data, bl.size, int(capacity),
                                      hot.ctypes.data if hot.size else None, pc.ctypes.data, pc.size,
                                      int(count_from), out.ctypes.data), "k3moe_trace_pin_sweep")
    return out


def hot_set(hist, n):
    """k3moe_hot_set: the n most frequent keys, hottest first, ties to the lower key."""
    h = np.ascontiguousarray(hist, np.uint32)
    out = np.zeros(int(n), np.int64)
    check(lib().k3moe_hot_set(h.ctypes.data, h.size, int(n), out.ctypes.data if n else None),
          "k3moe_hot_set")
    return out


def trace_save(path, keys, batch_len):
    keys, bl = _trace_arrays(keys, batch_len)
    check(lib().k3moe_trace_save(os.fsencode(path), keys.ctypes.data, bl.ctypes.data, bl.size),
          "k3moe_trace_save")


def trace_load(path):
    """k3moe_trace_load: (keys int64, batch_len int32)."""
    nk, nb = ctypes.c_int64(), ctypes.c_int32()
    p = os.fsencode(path)
    check(lib().k3moe_trace_load(p, None, 0, None, 0, ctypes.byref(nk), ctypes.byref(nb)),
          "k3moe_trace_load")
    keys = np.zeros(nk.value, np.int64)
    bl = np.zeros(nb.value, np.int32)
    check(lib().k3moe_trace_load(p, keys.ctypes.data, keys.size, bl.ctypes.data, bl.size,
                                 ctypes.byref(nk), ctypes.byref(nb)), "k3moe_trace_load")
    return keys, bl


def shared_expert_bytes(d, f):
    return lib().k3moe_shared_expert_bytes(d, f)


def shared_expert_view(blob_ptr, d, f):
    v = Bf16Expert()
    check(lib().k3moe_shared_expert_view(ctypes.byref(v), ctypes.c_void_p(blob_ptr), d, f),
          "k3moe_shared_expert_view")
    return v


def shared_workspace(n, f):
    return lib().k3moe_shared_workspace(n, f)


def shared_forward(out, x, T, views, d, f, workspace, accumulate=False, stream=None):
    """k3moe_shared_forward: out (+)= the shared experts `views` of x [T, d]."""
    n = len(views)
    arr = (Bf16Expert * n)(*views)
    nbytes = workspace.numel() * workspace.element_size()
    check(lib().k3moe_shared_forward(_ptr(out), _ptr(x), T, ctypes.cast(arr, ctypes.c_void_p), n, d, f,
                                     1 if accumulate else 0, _ptr(workspace), nbytes, _stream(stream)),
          "k3moe_shared_forward")


def stream_decode(layers, cache, X, T, out, eps=1e-6, stream=None, want_trace=True, trunk=None,
                  n_shared=0):
    """k3moe_stream_decode: T tokens through len(layers) layers over `cache`
    (and, with `trunk`, each layer's n_shared bf16 shared experts from it).
    Returns (ids [T, L, k], hits [T, L, k]) as numpy arrays when want_trace."""
    nl = len(layers)
    arr = (ctypes.c_void_p * nl)(*[l.h.value for l in layers])
    desc = StreamDesc(nl, ctypes.cast(arr, ctypes.c_void_p), cache.h.value, eps,
                      None if trunk is None else trunk.h.value, n_shared if trunk is not None else 0)
    kk = layers[0].k
    ids = np.zeros((T, nl, kk), np.int32) if want_trace else None
    hits = np.zeros((T, nl, kk), np.uint8) if want_trace else None
    check(lib().k3moe_stream_decode(ctypes.byref(desc), _ptr(X), T, _ptr(out),
                                    None if ids is None else ids.ctypes.data,
                                    None if hits is None else hits.ctypes.data, _stream(stream)),
          "k3moe_stream_decode")
    return ids, hits


def check_wait_timeout(stream=None):
    """k3moe_check_wait_timeout: enqueue the bounded-wait self-check."""
    check(lib().k3moe_check_wait_timeout(_stream(stream)), "k3moe_check_wait_timeout")
