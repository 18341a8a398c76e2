"""Plain fp64 CPU oracle of the activation-sparse decode FFN.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline arm are its only users; the CUDA library never loads it and it
never loads the CUDA library.  ctypes binding over ``oracle.c``; every
function here is marshalling only.  See ``oracle.h`` for what is computed
and which passage of the PowerInfer page each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DT = {"f16": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile liboracle.so next to the sources (gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i32, vp = ctypes.c_int32, ctypes.c_void_p
            L.or_decode_half.restype = ctypes.c_double
            L.or_decode_half.argtypes = [ctypes.c_uint16, i32]
            L.or_predict.restype = None
            L.or_predict.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, vp]
            L.or_compact.restype = i32
            L.or_compact.argtypes = [vp, i32, vp]
            L.or_union.restype = i32
            L.or_union.argtypes = [vp, i32, i32, vp, vp]
            L.or_hidden.restype = None
            L.or_hidden.argtypes = [i32, i32, i32, vp, vp, vp, vp, i32, vp]
            L.or_down.restype = None
            L.or_down.argtypes = [i32, i32, vp, vp, vp, i32, vp, vp]
            L.or_sparse_ffn.restype = None
            L.or_sparse_ffn.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, i32, vp, vp]
            L.or_dense_ffn.restype = None
            L.or_dense_ffn.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
            L.or_layer_decode.restype = i32
            L.or_layer_decode.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                          vp, vp, vp, vp]
            L.or_profile_counts.restype = None
            L.or_profile_counts.argtypes = [vp, i32, i32, vp]
            L.or_hot_order.restype = None
            L.or_hot_order.argtypes = [vp, i32, vp]
            L.or_permute_rows.restype = None
            L.or_permute_rows.argtypes = [vp, i32, i32, vp, vp]
            L.or_set_threads.restype = None
            L.or_set_threads.argtypes = [i32]
            L.or_get_threads.restype = i32
            L.or_get_threads.argtypes = []
            _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


def set_threads(n: int) -> None:
    lib().or_set_threads(int(n))


def get_threads() -> int:
    return lib().or_get_threads()


def decode_half(bits, dtype: str) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).ravel()
    f = lib().or_decode_half
    return np.array([f(int(v), _DT[dtype]) for v in b], dtype=np.float64)


def predict(layer, x):
    """u [batch, r], logits [batch, n] (fp64) for activations x [batch, d]."""
    x = _f32(np.atleast_2d(x))
    batch = x.shape[0]
    u = np.empty((batch, layer.r), np.float64)
    lg = np.empty((batch, layer.n), np.float64)
    lib().or_predict(layer.d, layer.n, layer.r, _DT[layer.dtype], _p(layer.A), _p(layer.Bm),
                     _p(layer.b1), _p(x), batch, _p(u), _p(lg))
    return u, lg


def compact(logits):
    """Ascending indices of the neurons with logit > 0."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    idx = np.empty(lg.shape[0], np.int32)
    c = lib().or_compact(_p(lg), lg.shape[0], _p(idx))
    return idx[:c].copy()


def union(logits):
    """(union indices, per-union-neuron token bitmask) of logits [batch, n]."""
    lg = np.ascontiguousarray(np.atleast_2d(logits), dtype=np.float64)
    batch, n = lg.shape
    uidx = np.empty(n, np.int32)
    mask = np.empty(n, np.uint32)
    c = lib().or_union(_p(lg), n, batch, _p(uidx), _p(mask))
    return uidx[:c].copy(), mask[:c].copy()


def hidden(layer, x, idx):
    x = _f32(np.ravel(x))
    idx = _i32(idx)
    h = np.empty(max(len(idx), 1), np.float64)
    lib().or_hidden(layer.d, _DT[layer.dtype], int(layer.gated), _p(layer.W1), _p(layer.b1),
                    _p(x), _p(idx), len(idx), _p(h))
    return h[:len(idx)]


def down(layer, idx, h):
    idx = _i32(idx)
    h = np.ascontiguousarray(h, dtype=np.float64)
    y = np.empty(layer.d, np.float64)
    lib().or_down(layer.d, _DT[layer.dtype], _p(layer.W2), _p(layer.b2), _p(idx), len(idx),
                  _p(h), _p(y))
    return y


def sparse_ffn(layer, x, idx):
    """y [d] (fp64) of one token over the listed neurons."""
    x = _f32(np.ravel(x))
    idx = _i32(idx)
    y = np.empty(layer.d, np.float64)
    lib().or_sparse_ffn(layer.d, _DT[layer.dtype], int(layer.gated), _p(layer.W1), _p(layer.b1),
                        _p(layer.W2), _p(layer.b2), _p(x), _p(idx), len(idx), _p(y), None)
    return y


def dense_ffn(layer, x):
    """y [d] (fp64) of one token over all neurons."""
    x = _f32(np.ravel(x))
    y = np.empty(layer.d, np.float64)
    lib().or_dense_ffn(layer.d, layer.n, _DT[layer.dtype], int(layer.gated), _p(layer.W1),
                       _p(layer.b1), _p(layer.W2), _p(layer.b2), _p(x), _p(y))
    return y


def layer_decode(layer, x, residual: bool = False):
    """One decode step of one token: (logits, idx, y, x_next or None)."""
    x = _f32(np.ravel(x))
    lg = np.empty(layer.n, np.float64)
    idx = np.empty(layer.n, np.int32)
    y = np.empty(layer.d, np.float64)
    xn = np.empty(layer.d, np.float32) if residual else None
    c = lib().or_layer_decode(layer.d, layer.n, layer.r, _DT[layer.dtype], int(layer.gated),
                              _p(layer.A), _p(layer.Bm), _p(layer.b1), _p(layer.W1),
                              _p(layer.W2), _p(layer.b2), _p(x), _p(lg), _p(idx), _p(y), _p(xn))
    return lg, idx[:c].copy(), y, xn


# ------------------------------------------------------------ offline placement
def profile_counts(logits, counts=None):
    """Activation counts per neuron over the tokens of logits [batch, n]
    (added to counts if given): the profiler of the page's "Offline
    Section"."""
    lg = np.ascontiguousarray(np.atleast_2d(logits), dtype=np.float64)
    batch, n = lg.shape
    c = np.zeros(n, np.uint32) if counts is None else np.ascontiguousarray(counts, np.uint32)
    lib().or_profile_counts(_p(lg), n, batch, _p(c))
    return c


def hot_order(counts):
    """perm[k] = original neuron placed at position k: more activations
    first, equal counts in ascending index (the neuron table)."""
    c = np.ascontiguousarray(counts, np.uint32)
    perm = np.empty(c.shape[0], np.int32)
    lib().or_hot_order(_p(c), c.shape[0], _p(perm))
    return perm


def permute_rows(rows, perm):
    """Row k of the result = row perm[k] of rows (any dtype, one row per
    neuron)."""
    src = np.ascontiguousarray(rows)
    dst = np.empty_like(src)
    n = src.shape[0]
    rb = src.nbytes // max(n, 1)
    lib().or_permute_rows(_p(src), n, rb, _p(np.ascontiguousarray(perm, np.int32)), _p(dst))
    return dst
