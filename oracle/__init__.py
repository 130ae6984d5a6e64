"""fp64 CPU oracle for the paged KV-cache write and paged decode attention.

TEST INFRASTRUCTURE ONLY.  The product (the CUDA library and its binding)
never imports this package; only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg do.  It shares no code with the
CUDA path.  The arithmetic lives in ``oracle.c`` (plain C, fp64, no
fast-math); this module compiles it with gcc and marshals numpy arrays.

Element dtype tags: "f32", "bf16" (uint16 bit patterns), "f16" (uint16 bit
patterns), "e4m3" (uint8 codes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_DT = {"f32": 0, "bf16": 1, "f16": 2, "e4m3": 3}
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, dbl, flt = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
            L.orc_e4m3_decode.restype = dbl
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [flt]
            L.orc_quantize_e4m3.restype = ctypes.c_uint8
            L.orc_quantize_e4m3.argtypes = [flt, flt]
            L.orc_write_flat.restype = i32
            L.orc_write_flat.argtypes = [P, i32, i64, i64, i32, i32, P, i64, P, i32, flt]
            L.orc_dense_decode.restype = i32
            L.orc_dense_decode.argtypes = [P, P, P, i64, i32, i32, i32, dbl, P, P]
            L.orc_partial_decode.restype = i32
            L.orc_partial_decode.argtypes = [P, P, P, i64, i64, i32, i32, i32, dbl, P, P, P]
            L.orc_lse_merge.restype = None
            L.orc_lse_merge.argtypes = [P, P, P, i32, i32, P]
            L.orc_write_flat_heads.restype = i32
            L.orc_write_flat_heads.argtypes = [P, i32, i64, i64, i32, i32, P, i64, P, i32, P]
            L.orc_attention_causal.restype = i32
            L.orc_attention_causal.argtypes = [P, P, P, i64, i64, i32, i32, i32, dbl, P, P]
            L.orc_paged_walk_decode.restype = i32
            L.orc_paged_walk_decode.argtypes = [P, P, P, P, i32, i64, i32, i32, i32, dbl, P]
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


# ---------------------------------------------------------------- E4M3 codec

def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8)
    L = lib()
    return np.array([L.orc_e4m3_decode(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float32)
    L = lib()
    return np.array([L.orc_e4m3_encode(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def quantize_e4m3(x, scale: float) -> np.ndarray:
    a = np.asarray(x, dtype=np.float32)
    L = lib()
    s = float(np.float32(scale))
    return np.array([L.orc_quantize_e4m3(float(v), s) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


# --------------------------------------------------------------------- write

def write_flat(rows: np.ndarray, rows_dtype: str, slots: np.ndarray, cache_flat: np.ndarray,
               cache_dtype: str, scale=1.0) -> None:
    """rows [T, Hkv, D] (or a view with a token stride); cache_flat [num_slots, Hkv, D].

    scale: one fp32 scale, or a sequence of Hkv per-head scales (head h quantises with
    scale[h]).  Writes in place.  Raises on a slot >= num_slots.
    """
    assert rows.ndim == 3 and cache_flat.ndim == 3
    assert rows.strides[2] == rows.itemsize and rows.strides[1] == rows.shape[2] * rows.itemsize
    assert cache_flat.flags.c_contiguous
    T, Hkv, D = rows.shape
    assert cache_flat.shape[1:] == (Hkv, D)
    row_stride = rows.strides[0] // rows.itemsize
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    assert sl.shape == (T,)
    args = (rows.ctypes.data_as(ctypes.c_void_p), _DT[rows_dtype], T, row_stride, Hkv, D,
            _ptr(sl), cache_flat.shape[0], _ptr(cache_flat), _DT[cache_dtype])
    if np.ndim(scale) == 0:
        rc = lib().orc_write_flat(*args, float(np.float32(scale)))
    else:
        sc = np.ascontiguousarray(scale, dtype=np.float32)
        assert sc.shape == (Hkv,)
        rc = lib().orc_write_flat_heads(*args, _ptr(sc))
    if rc != 0:
        raise ValueError("orc_write_flat failed with %d" % rc)


# -------------------------------------------------------------------- decode

def dense_decode(q, K, V, scale: float, return_probs: bool = False):
    """One sequence: q [Hq, D], K/V [L, Hkv, D] in logical order -> out [Hq, D] (fp64)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    Hq, D = q.shape
    L, Hkv, D2 = K.shape
    assert D2 == D and V.shape == K.shape
    out = np.zeros((Hq, D), dtype=np.float64)
    probs = np.zeros((Hq, L), dtype=np.float64) if return_probs else None
    rc = lib().orc_dense_decode(_ptr(q), _ptr(K), _ptr(V), L, Hq, Hkv, D, float(scale), _ptr(out),
                                _ptr(probs) if probs is not None else None)
    if rc != 0:
        raise ValueError("orc_dense_decode failed with %d" % rc)
    return (out, probs) if return_probs else out


def attention_causal(q, K, V, scale: float, alibi_slopes=None) -> np.ndarray:
    """n query tokens of one sequence: q [n, Hq, D], K/V [L, Hkv, D] -> out [n, Hq, D] (fp64).
    Query i sits at position L - n + i and sees tokens 0 .. L - n + i; alibi_slopes [Hq]
    adds slope_h * (t - (L - n + i)) to the logits."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    n, Hq, D = q.shape
    L, Hkv, D2 = K.shape
    assert D2 == D and V.shape == K.shape
    sl = None if alibi_slopes is None else _f64(alibi_slopes)
    out = np.zeros((n, Hq, D), dtype=np.float64)
    rc = lib().orc_attention_causal(_ptr(q), _ptr(K), _ptr(V), n, L, Hq, Hkv, D, float(scale),
                                    _ptr(sl) if sl is not None else None, _ptr(out))
    if rc != 0:
        raise ValueError("orc_attention_causal failed with %d" % rc)
    return out


def partial_decode(q, K, V, t0: int, t1: int, scale: float):
    """Split-KV state of tokens [t0, t1): (m [Hq], l [Hq], acc [Hq, D])."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    Hq, D = q.shape
    Hkv = K.shape[1]
    m = np.zeros(Hq)
    l = np.zeros(Hq)
    acc = np.zeros((Hq, D))
    rc = lib().orc_partial_decode(_ptr(q), _ptr(K), _ptr(V), t0, t1, Hq, Hkv, D, float(scale),
                                  _ptr(m), _ptr(l), _ptr(acc))
    if rc != 0:
        raise ValueError("orc_partial_decode failed with %d" % rc)
    return m, l, acc


def lse_merge(m, l, acc) -> np.ndarray:
    """Merge P partial states of one head: m [P], l [P], acc [P, D] -> out [D]."""
    m, l, acc = _f64(m), _f64(l), _f64(acc)
    P, D = acc.shape
    out = np.zeros(D)
    lib().orc_lse_merge(_ptr(m), _ptr(l), _ptr(acc), P, D, _ptr(out))
    return out


def paged_walk_decode(q, pool_k, pool_v, block_table_row, block_size: int, L: int, scale: float):
    """Walk a block-table row over flat-slot pools [num_slots, Hkv, D] -> out [Hq, D]."""
    q, pk, pv = _f64(q), _f64(pool_k), _f64(pool_v)
    Hq, D = q.shape
    Hkv = pk.shape[1]
    bt = np.ascontiguousarray(block_table_row, dtype=np.int32)
    out = np.zeros((Hq, D))
    rc = lib().orc_paged_walk_decode(_ptr(q), _ptr(pk), _ptr(pv), _ptr(bt), block_size, L, Hq, Hkv, D,
                                     float(scale), _ptr(out))
    if rc != 0:
        raise ValueError("orc_paged_walk_decode failed with %d" % rc)
    return out


# ------------------------------------------------------- cache element values

def cache_values(cache_flat: np.ndarray, cache_dtype: str, scale=1.0) -> np.ndarray:
    """Element values of a flat cache [n, Hkv, D] in fp64 (E4M3 codes are decoded and multiplied
    by the scale: one fp32 value, or Hkv per-head values)."""
    if cache_dtype == "f32":
        return cache_flat.astype(np.float64)
    if cache_dtype == "bf16":
        return (cache_flat.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if cache_dtype == "f16":
        return cache_flat.view(np.float16).astype(np.float64)
    if cache_dtype == "e4m3":
        table = e4m3_decode(np.arange(256, dtype=np.uint8))
        if np.ndim(scale) == 0:
            return table[cache_flat] * float(np.float32(scale))
        sc = np.asarray(scale, dtype=np.float32).astype(np.float64)
        return table[cache_flat] * sc.reshape((1, -1) + (1,) * (cache_flat.ndim - 2))
    raise ValueError(cache_dtype)
