"""ctypes front end of the fp32 contract emulator (``contract_emulator.c``).

TEST INFRASTRUCTURE ONLY.  Given fp32 logits, it reproduces the contract's
tile partials, shard records, log-sum-exp and logprob bit for bit.  The
tests feed it logits that are known exactly on the CPU (``exact_case``
inputs), never values read back from the GPU.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        f, i64, i32 = ctypes.c_float, ctypes.c_int64, ctypes.c_int
        P = ctypes.c_void_p
        L.emu_exp.restype = f
        L.emu_exp.argtypes = [f]
        L.emu_log.restype = f
        L.emu_log.argtypes = [f]
        L.emu_merge.restype = None
        L.emu_merge.argtypes = [f, f, f, f, P, P]
        L.emu_tile_ms.restype = None
        L.emu_tile_ms.argtypes = [P, i32, P, P]
        L.emu_tree.restype = None
        L.emu_tree.argtypes = [P, P, i64, P, P]
        L.emu_tree_nodes.restype = i32
        L.emu_tree_nodes.argtypes = [i64, i32, P, P]
        L.emu_tile_partials.restype = None
        L.emu_tile_partials.argtypes = [P, i64, i64, P, P]
        L.emu_linear_logprob.restype = i32
        L.emu_linear_logprob.argtypes = [P, i64, i64, P, P, i32, P, P, P, P, P, P, P, P]
        for name in ("emu_exp_sweep", "emu_log_sweep"):
            fn = getattr(L, name)
            fn.restype = None
            fn.argtypes = [f, f, P, P, P]
        L.emu_log_softmax.restype = i32
        L.emu_log_softmax.argtypes = [P, i64, i64, P, P, P]
        L.emu_grad_logits.restype = None
        L.emu_grad_logits.argtypes = [P, i64, i64, P, P, P, P, P]
        L.emu_rsqrt.restype = f
        L.emu_rsqrt.argtypes = [f]
        L.emu_rsqrt_sweep.restype = None
        L.emu_rsqrt_sweep.argtypes = [f, f, P, P, P]
        L.emu_rmsnorm.restype = None
        L.emu_rmsnorm.argtypes = [P, P, P, f, i64, i64, P, P]
        L.emu_constants.restype = None
        L.emu_constants.argtypes = [P]
        L.emu_primitive_hash.restype = ctypes.c_uint64
        L.emu_primitive_hash.argtypes = [i32, ctypes.c_uint32, ctypes.c_uint64]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def primitive_hash(which: str, first: int, count: int) -> int:
    """sum_i (bits(f(x_i)) + 0x9E3779B9) (2 i + 1) mod 2^64 over the fp32 bit patterns
    [first, first + count) for f = exp ("exp" and "exp_x2"), log or rsqrt."""
    code = {"exp": 0, "exp_x2": 1, "log": 2, "rsqrt": 3}[which]
    return int(lib().emu_primitive_hash(code, first, count))


def exp(x: float) -> np.float32:
    return np.float32(lib().emu_exp(ctypes.c_float(x)))


def log(x: float) -> np.float32:
    return np.float32(lib().emu_log(ctypes.c_float(x)))


def merge(m1, s1, m2, s2):
    mo, so = ctypes.c_float(), ctypes.c_float()
    lib().emu_merge(m1, s1, m2, s2, ctypes.byref(mo), ctypes.byref(so))
    return np.float32(mo.value), np.float32(so.value)


def tile_ms(v: np.ndarray):
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert 1 <= v.shape[0] <= 128
    mo, so = ctypes.c_float(), ctypes.c_float()
    lib().emu_tile_ms(_ptr(v), int(v.shape[0]), ctypes.byref(mo), ctypes.byref(so))
    return np.float32(mo.value), np.float32(so.value)


def tree(m: np.ndarray, s: np.ndarray):
    m = np.ascontiguousarray(m, dtype=np.float32)
    s = np.ascontiguousarray(s, dtype=np.float32)
    mo, so = ctypes.c_float(), ctypes.c_float()
    lib().emu_tree(_ptr(m), _ptr(s), int(m.shape[0]), ctypes.byref(mo), ctypes.byref(so))
    return np.float32(mo.value), np.float32(so.value)


def tree_nodes(n_tiles: int, depth: int):
    b = np.zeros(64, dtype=np.int64)
    e = np.zeros(64, dtype=np.int64)
    rc = lib().emu_tree_nodes(n_tiles, depth, _ptr(b), _ptr(e))
    if rc != 0:
        raise ValueError("tree too shallow")
    k = 1 << depth
    return list(zip(b[:k].tolist(), e[:k].tolist()))


def tile_partials(logits: np.ndarray):
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, V = L.shape
    nt = (V + 127) // 128
    tm = np.empty((T, nt), dtype=np.float32)
    ts = np.empty((T, nt), dtype=np.float32)
    lib().emu_tile_partials(_ptr(L), T, V, _ptr(tm), _ptr(ts))
    return tm, ts


def linear_logprob(logits: np.ndarray, targets: np.ndarray, active: Optional[np.ndarray] = None,
                   n_shards: int = 1):
    """Contract outputs from fp32 logits [T, V].

    Returns a dict: logprob, lse [T]; rec_m, rec_s, rec_tgt [n_shards, T];
    rec_owned (uint32) [n_shards, T]; root_m, root_s [T] (tree taken
    directly over all tiles, without the shard level).
    """
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, V = L.shape
    tg = np.ascontiguousarray(targets, dtype=np.int32)
    act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
    out = {
        "logprob": np.empty(T, np.float32), "lse": np.empty(T, np.float32),
        "rec_m": np.empty((n_shards, T), np.float32), "rec_s": np.empty((n_shards, T), np.float32),
        "rec_tgt": np.empty((n_shards, T), np.float32),
        "rec_owned": np.empty((n_shards, T), np.uint32),
        "root_m": np.empty(T, np.float32), "root_s": np.empty(T, np.float32),
    }
    rc = lib().emu_linear_logprob(_ptr(L), T, V, _ptr(tg), _ptr(act), n_shards,
                                  _ptr(out["logprob"]), _ptr(out["lse"]),
                                  _ptr(out["rec_m"]), _ptr(out["rec_s"]), _ptr(out["rec_tgt"]),
                                  _ptr(out["rec_owned"]), _ptr(out["root_m"]), _ptr(out["root_s"]))
    if rc != 0:
        raise ValueError("unsupported shard count %d for V=%d" % (n_shards, V))
    return out


def log_softmax(logits: np.ndarray, active: Optional[np.ndarray] = None):
    """Contract log_softmax of fp32 logits [T, V] -> (out [T, V], lse [T])."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, V = L.shape
    act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
    out = np.empty((T, V), np.float32)
    lse = np.empty(T, np.float32)
    rc = lib().emu_log_softmax(_ptr(L), T, V, _ptr(act), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("emu_log_softmax failed")
    return out, lse


def grad_logits(logits: np.ndarray, lse: np.ndarray, targets: np.ndarray, grad: np.ndarray,
                active: Optional[np.ndarray] = None) -> np.ndarray:
    """bf16 bits [T, V] of g * (onehot - exp(l - lse)) as the backward's first stage forms it."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, V = L.shape
    out = np.empty((T, V), np.uint16)
    act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
    lib().emu_grad_logits(_ptr(L), T, V, _ptr(np.ascontiguousarray(lse, np.float32)),
                          _ptr(np.ascontiguousarray(targets, np.int32)),
                          _ptr(np.ascontiguousarray(grad, np.float32)), _ptr(act), _ptr(out))
    return out


def exp_sweep(lo: float, hi: float):
    mu, wx, cnt = ctypes.c_double(), ctypes.c_float(), ctypes.c_int64()
    lib().emu_exp_sweep(lo, hi, ctypes.byref(mu), ctypes.byref(wx), ctypes.byref(cnt))
    return mu.value, wx.value, cnt.value


def log_sweep(lo: float, hi: float):
    mu, wx, cnt = ctypes.c_double(), ctypes.c_float(), ctypes.c_int64()
    lib().emu_log_sweep(lo, hi, ctypes.byref(mu), ctypes.byref(wx), ctypes.byref(cnt))
    return mu.value, wx.value, cnt.value


def constants():
    out = np.zeros(16, dtype=np.float32)
    lib().emu_constants(_ptr(out))
    names = ["log2e", "ln2_hi", "ln2_lo", "shifter", "sqrt2"] + ["inv_fact%d" % k for k in range(8)] \
        + ["two_thirds", "two_fifths", "two_elevenths"]
    return dict(zip(names, out.tolist()))


def exact_fp32_logits(logits_f64: np.ndarray) -> np.ndarray:
    """Cast fp64 logits to fp32, asserting the cast is exact (exact_case inputs)."""
    L32 = logits_f64.astype(np.float32)
    if not np.array_equal(L32.astype(np.float64), logits_f64):
        raise ValueError("logits are not exactly representable in fp32")
    return L32



def rsqrt(x: float) -> np.float32:
    return np.float32(lib().emu_rsqrt(ctypes.c_float(x)))


def rsqrt_sweep(lo: float, hi: float):
    mu, wx, cnt = ctypes.c_double(), ctypes.c_float(), ctypes.c_int64()
    lib().emu_rsqrt_sweep(lo, hi, ctypes.byref(mu), ctypes.byref(wx), ctypes.byref(cnt))
    return mu.value, wx.value, cnt.value


def rmsnorm(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float,
            residual_bits: Optional[np.ndarray] = None):
    """Contract RMSNorm -> (y bf16 bits [T, H], x' bf16 bits [T, H] or None)."""
    x = np.ascontiguousarray(x_bits, np.uint16)
    T, H = x.shape
    g = np.ascontiguousarray(gamma_bits, np.uint16)
    r = None if residual_bits is None else np.ascontiguousarray(residual_bits, np.uint16)
    y = np.empty((T, H), np.uint16)
    xr = None if r is None else np.empty((T, H), np.uint16)
    lib().emu_rmsnorm(_ptr(x), _ptr(r), _ptr(g), ctypes.c_float(eps), T, H, _ptr(y), _ptr(xr))
    return y, xr
