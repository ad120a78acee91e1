"""Seeded synthetic inputs for the MXFP4 routed-expert MoE layer.

This module is shared by the oracle tests, the GPU parity tests and
``bench.py``.  It holds none of the method's arithmetic: it only draws random
numbers (SplitMix64 in counter mode, see ``k3synth.c``) in the shapes and
distributions of the workloads:

* packed MXFP4 matrices in the canonical layout of the explainer page
  ("kimi-k3-in-c", ai.thesatyajit.com, section "Reduction one"): a nibble
  plane ``[rows][in/2]`` of uniform random bytes (so every 4-bit E2M1 code is
  uniform in 0..15) and an E8M0 plane ``[rows][in/32]`` uniform in
  ``[e_lo, e_hi]`` (120..130 by default);
* activations ``x ~ N(0, 1)`` rounded to fp32 (or bf16), one substream per
  token so a single token can be redrawn on its own;
* router weights ``W_r ~ N(0, 0.02)`` rounded to bf16;
* a per-expert selection bias: ``N(0, 1)`` in fp32, or a Zipf(s) log-weight
  ``-s * ln(rank)`` over a seeded permutation of ranks;
* bf16 shared experts with unit-variance products (gate/up ~ N(0, 1/sqrt(d)),
  down ~ N(0, 1/sqrt(f))).

Every tensor is addressed by a 64-bit tag (kind, pool, layer, index,
substream) under the base seed, so any one expert can be regenerated without
the others.
"""
import ctypes
import os
import subprocess

import numpy as np

BASE_SEED = 0x4B334D4F

# tensor kinds
K_GATE_PACKED, K_GATE_SCALES = 1, 2
K_UP_PACKED, K_UP_SCALES = 3, 4
K_DOWN_PACKED, K_DOWN_SCALES = 5, 6
K_TOKEN = 7
K_ROUTER = 8
K_BIAS_NORMAL = 9
K_ZIPF_PERM = 10
K_MISC = 11
K_SHARED_GATE, K_SHARED_UP, K_SHARED_DOWN = 12, 13, 14

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3synth.c")
_SO = os.path.join(_HERE, "libk3synth.so")
_lib = None


def build(force=False):
    """Compile the generator with gcc (plain C, no architecture flags)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, sz, p = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p
        L.k3s_key.restype = u64
        L.k3s_key.argtypes = [u64, u64]
        L.k3s_u64.restype = u64
        L.k3s_u64.argtypes = [u64, u64]
        L.k3s_bytes.argtypes = [p, sz, u64]
        L.k3s_uniform_u8.argtypes = [p, sz, u64, ctypes.c_int, ctypes.c_int]
        L.k3s_normal_f64.argtypes = [p, sz, u64, ctypes.c_double, ctypes.c_double]
        L.k3s_normal_f32.argtypes = [p, sz, u64, ctypes.c_double, ctypes.c_double]
        L.k3s_normal_bf16.argtypes = [p, sz, u64, ctypes.c_double, ctypes.c_double]
        L.k3s_permutation.argtypes = [p, ctypes.c_int, u64]
        _lib = L
    return _lib


def tag(kind, pool=0, layer=0, index=0, sub=0):
    assert 0 <= kind < 256 and 0 <= pool < 256 and 0 <= layer < 256
    assert 0 <= index < (1 << 24) and 0 <= sub < (1 << 16)
    return (kind << 56) | (pool << 48) | (layer << 40) | (index << 16) | sub


def key(t, seed=BASE_SEED):
    return lib().k3s_key(seed, t)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def fill_bytes(out, t, seed=BASE_SEED):
    out = np.ascontiguousarray(out)
    lib().k3s_bytes(_ptr(out), out.nbytes, key(t, seed))
    return out


def fill_uniform_u8(out, t, lo, hi, seed=BASE_SEED):
    lib().k3s_uniform_u8(_ptr(out), out.size, key(t, seed), lo, hi)
    return out


def normal_f32(shape, t, mean=0.0, std=1.0, seed=BASE_SEED):
    out = np.empty(shape, np.float32)
    lib().k3s_normal_f32(_ptr(out), out.size, key(t, seed), mean, std)
    return out


def normal_f64(shape, t, mean=0.0, std=1.0, seed=BASE_SEED):
    out = np.empty(shape, np.float64)
    lib().k3s_normal_f64(_ptr(out), out.size, key(t, seed), mean, std)
    return out


def normal_bf16(shape, t, mean=0.0, std=1.0, seed=BASE_SEED):
    """bf16 bit patterns (uint16) of N(mean, std) draws."""
    out = np.empty(shape, np.uint16)
    lib().k3s_normal_bf16(_ptr(out), out.size, key(t, seed), mean, std)
    return out


def permutation(n, t, seed=BASE_SEED):
    out = np.empty(n, np.int32)
    lib().k3s_permutation(_ptr(out), n, key(t, seed))
    return out


# ---------------------------------------------------------------- workloads

def matrix(kind_packed, kind_scales, rows, cols, pool, layer, expert, e_lo=120, e_hi=130,
           seed=BASE_SEED):
    """One packed MXFP4 matrix in canonical layout: (packed [rows, cols/2] u8,
    scales [rows, cols/32] u8)."""
    assert cols % 32 == 0
    packed = np.empty((rows, cols // 2), np.uint8)
    fill_bytes(packed, tag(kind_packed, pool, layer, expert), seed)
    scales = np.empty((rows, cols // 32), np.uint8)
    fill_uniform_u8(scales, tag(kind_scales, pool, layer, expert), e_lo, e_hi, seed)
    return packed, scales


def expert(pool, layer, e, d=7168, f=1536, e_lo=120, e_hi=130, seed=BASE_SEED):
    """Planes of one expert: gate/up [f x d], down [d x f] (rows x input)."""
    gp, gs = matrix(K_GATE_PACKED, K_GATE_SCALES, f, d, pool, layer, e, e_lo, e_hi, seed)
    up, us = matrix(K_UP_PACKED, K_UP_SCALES, f, d, pool, layer, e, e_lo, e_hi, seed)
    dp, ds = matrix(K_DOWN_PACKED, K_DOWN_SCALES, d, f, pool, layer, e, e_lo, e_hi, seed)
    return dict(gate_packed=gp, gate_scales=gs, up_packed=up, up_scales=us,
                down_packed=dp, down_scales=ds, d=d, f=f)


def shared_expert(pool, layer, s, d=7168, f=1536, seed=BASE_SEED):
    """One bf16 shared expert (bit patterns): gate, up [f x d] ~ N(0, 1/sqrt(d)),
    down [d x f] ~ N(0, 1/sqrt(f)) (unit-variance products)."""
    return dict(gate=normal_bf16((f, d), tag(K_SHARED_GATE, pool, layer, s), 0.0, d ** -0.5, seed),
                up=normal_bf16((f, d), tag(K_SHARED_UP, pool, layer, s), 0.0, d ** -0.5, seed),
                down=normal_bf16((d, f), tag(K_SHARED_DOWN, pool, layer, s), 0.0, f ** -0.5, seed),
                d=d, f=f)


def token_f32(pool, t, d=7168, sub=0, seed=BASE_SEED):
    """Activation row of token t drawn from substream `sub`: x ~ N(0,1), fp32."""
    return normal_f32((d,), tag(K_TOKEN, pool, 0, t, sub), 0.0, 1.0, seed)


def token_bf16(pool, t, d=7168, sub=0, seed=BASE_SEED):
    return normal_bf16((d,), tag(K_TOKEN, pool, 0, t, sub), 0.0, 1.0, seed)


def tokens_f32(pool, T, d=7168, subs=None, t0=0, seed=BASE_SEED):
    subs = np.zeros(T, np.int64) if subs is None else subs
    return np.stack([token_f32(pool, t0 + i, d, int(subs[i]), seed) for i in range(T)])


def tokens_bf16(pool, T, d=7168, subs=None, t0=0, seed=BASE_SEED):
    subs = np.zeros(T, np.int64) if subs is None else subs
    return np.stack([token_bf16(pool, t0 + i, d, int(subs[i]), seed) for i in range(T)])


def router_bf16(pool, layer, E=896, d=7168, std=0.02, seed=BASE_SEED):
    """Router weight W_r [E x d] as bf16 bit patterns, N(0, std)."""
    return normal_bf16((E, d), tag(K_ROUTER, pool, layer), 0.0, std, seed)


def bias_normal(pool, layer, E=896, seed=BASE_SEED):
    """Per-expert selection bias ~ N(0, 1), fp32."""
    return normal_f32((E,), tag(K_BIAS_NORMAL, pool, layer), 0.0, 1.0, seed)


def bias_zipf(pool, layer, E=896, s=1.1, seed=BASE_SEED):
    """Per-expert selection bias -s*ln(rank), rank a seeded permutation of 1..E,
    rounded to fp32: the log of a Zipf(s) popularity weight."""
    rank = permutation(E, tag(K_ZIPF_PERM, pool, layer), seed).astype(np.float64) + 1.0
    return (-s * np.log(rank)).astype(np.float32)
