"""activation_sparse_decode_rank_gb300 — activation-sparse decode FFN on GB300.

Thin ctypes binding of libpi.so (C ABI in include/pi.h).  Each ``pi_*``
function here has the name and argument order of the C entry point and only
marshals arguments: torch tensors become device pointers, streams become
``cudaStream_t`` handles.  Every step of the computation runs in the CUDA
kernels of libpi; there is no Python or CPU fallback, and importing the
library fails loudly if libpi.so has not been built.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
_LIB = os.path.join(_HERE, "libpi.so")
_lock = threading.Lock()
_lib = None

PI_OK, PI_ERR_NULL, PI_ERR_SHAPE, PI_ERR_DTYPE, PI_ERR_ALIGN, PI_ERR_WORKSPACE, \
    PI_ERR_CAPACITY, PI_ERR_LAUNCH, PI_ERR_TIMEOUT, PI_ERR_CUDA, PI_ERR_INDEX, PI_ERR_RANGE, \
    PI_ERR_CAPTURE = range(13)
PI_F16, PI_BF16 = 0, 1
PI_LAYOUT_SPLIT, PI_LAYOUT_PACKED = 0, 1

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared"]


def _sources():
    srcs = [os.path.join(_CSRC, f) for f in sorted(os.listdir(_CSRC))
            if f.endswith((".cu", ".cuh"))]
    return srcs + [os.path.join(_INCLUDE, "pi.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libpi.so in-tree for sm_103a with nvcc."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in _sources())
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["nvcc", *NVCC_FLAGS, "-o", tmp, os.path.join(_CSRC, "pi_abi.cu")]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class PiError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class pi_ffn_desc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n", ctypes.c_int32), ("r", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("gated", ctypes.c_int32),
                ("hot_prefix", ctypes.c_int32), ("layout", ctypes.c_int32)]


class pi_layer_weights(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("Bm", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("W1", ctypes.c_void_p), ("W2", ctypes.c_void_p), ("b2", ctypes.c_void_p)]


PI_PATH_FUSED, PI_PATH_PER_TOKEN, PI_PATH_UNION, PI_PATH_DENSE = range(4)
PI_PATHS, PI_COST_TIERS = 4, 4
PATH_NAMES = ("fused", "per_token", "union", "dense")


class pi_cost_model(ctypes.Structure):
    _fields_ = [("tier_max_batch", ctypes.c_int32 * PI_COST_TIERS),
                ("fixed_us", (ctypes.c_double * PI_COST_TIERS) * PI_PATHS),
                ("gbs", (ctypes.c_double * PI_COST_TIERS) * PI_PATHS)]


class pi_plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("est_us", ctypes.c_double * PI_PATHS),
                ("bytes", ctypes.c_double * PI_PATHS), ("active_rows", ctypes.c_double),
                ("union_rows", ctypes.c_double)]


# Names and argument lists of the C entry points (include/pi.h).
_P, _I32, _SZ, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_int64
_DESC = ctypes.POINTER(pi_ffn_desc)
_W = ctypes.POINTER(pi_layer_weights)
SIGNATURES = {
    "pi_workspace_size": (ctypes.c_size_t, [_DESC, _I32]),
    "pi_predict": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _I32, _P, _P, _SZ, _P]),
    "pi_compact": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "pi_sparse_ffn": (ctypes.c_int, [_DESC, _W, _P, _I32, _P, _P, _I32, _P, _P, _P, _P, _P, _P,
                                     _SZ, _P]),
    "pi_dense_ffn": (ctypes.c_int, [_DESC, _W, _P, _I32, _P, _P, _SZ, _P]),
    "pi_layer_decode": (ctypes.c_int, [_DESC, _W, _P, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "pi_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pi_selftest_wait_timeout": (ctypes.c_int, [_P, _P, _SZ, _I64, _P]),
    "pi_selftest_ring_timeout": (ctypes.c_int, [_DESC, _W, _P, _P, _P, _I32, _P, _P, _P, _SZ,
                                                _I64, _P]),
    "pi_pack_weights": (ctypes.c_int, [_DESC, _P, _P, _P, _P]),
    "pi_layer_decode_static": (ctypes.c_int, [_DESC, _W, _P, _P, _P, _P, _P, _P, _P]),
    "pi_decode_layers": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P, _SZ,
                                        _P]),
    "pi_profile_counts": (ctypes.c_int, [_P, _I32, _I32, _P, _P]),
    "pi_hot_order": (ctypes.c_int, [_P, _I32, _P, _P]),
    "pi_permute_neurons": (ctypes.c_int, [_DESC, _W, _P, _W, _P, _P]),
    "pi_default_cost_model": (None, [ctypes.POINTER(pi_cost_model)]),
    "pi_plan_dispatch": (ctypes.c_int, [_DESC, _I32, ctypes.POINTER(ctypes.c_float),
                                        ctypes.c_float, _I32, ctypes.POINTER(pi_cost_model),
                                        ctypes.POINTER(pi_plan)]),
    "pi_decode_planned": (ctypes.c_int, [_DESC, _W, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _SZ,
                                         _P]),
    "pi_decoder_create": (ctypes.c_int, [_DESC, _W, ctypes.POINTER(ctypes.c_float),
                                         ctypes.c_float, _I32, ctypes.POINTER(pi_cost_model),
                                         _P, _P, _P, _P, _P, _SZ, ctypes.POINTER(_P)]),
    "pi_decoder_run": (ctypes.c_int, [_P, _I32, _P]),
    "pi_decoder_plan": (ctypes.c_int, [_P, _I32, ctypes.POINTER(pi_plan)]),
    "pi_decoder_destroy": (None, [_P]),
    "pi_shard_desc": (ctypes.c_int, [_DESC, _I32, _I32, _DESC]),
    "pi_shard_layer": (ctypes.c_int, [_DESC, _W, _I32, _I32, _W, _P]),
    "pi_shard_reduce": (ctypes.c_int, [_P, _I32, _I32, _I32, _P, _P, _P]),
}


def lib():
    """The loaded libpi.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB):
                raise RuntimeError(
                    f"libpi.so not found at {_LIB}: build it first "
                    "(activation_sparse_decode_rank_gb300.build())")
            L = ctypes.CDLL(_LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


# ------------------------------------------------------------ marshalling
def _ptr(t):
    """Device pointer of a torch tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def status_string(status: int) -> str:
    return lib().pi_status_string(int(status)).decode()


def check(status: int, where: str = "libpi") -> None:
    if status != PI_OK:
        raise PiError(status, where)


def make_desc(d: int, n: int, r: int, dtype: str = "f16", gated: bool = False,
              hot_prefix: int = 0, packed: bool = False) -> pi_ffn_desc:
    return pi_ffn_desc(d, n, r, PI_BF16 if dtype == "bf16" else PI_F16, int(gated), hot_prefix,
                       PI_LAYOUT_PACKED if packed else PI_LAYOUT_SPLIT)


def make_weights(A, Bm, b1, W1, W2, b2=None) -> pi_layer_weights:
    return pi_layer_weights(_ptr(A), _ptr(Bm), _ptr(b1), _ptr(W1), _ptr(W2), _ptr(b2))


def pi_workspace_size(desc: pi_ffn_desc, batch: int) -> int:
    return lib().pi_workspace_size(ctypes.byref(desc), batch)


def workspace(desc: pi_ffn_desc, batch: int, device="cuda"):
    """A zero-filled workspace tensor of pi_workspace_size(desc, batch) bytes."""
    import torch
    nbytes = pi_workspace_size(desc, batch)
    if nbytes == 0:
        raise PiError(PI_ERR_SHAPE, "pi_workspace_size")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def pi_predict(desc, A, Bm, b1, x, batch, logits, ws, ws_bytes=None, stream=None) -> int:
    return lib().pi_predict(ctypes.byref(desc), _ptr(A), _ptr(Bm), _ptr(b1), _ptr(x), batch,
                            _ptr(logits), _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes,
                            _stream(stream))


def pi_compact(logits, n, batch, idx, cnt, cap, union_idx, union_cnt, tok_mask, dev_status, ws,
               ws_bytes=None, stream=None) -> int:
    wsb = (ws.numel() if ws is not None else 0) if ws_bytes is None else ws_bytes
    return lib().pi_compact(_ptr(logits), n, batch, _ptr(idx), _ptr(cnt), cap, _ptr(union_idx),
                            _ptr(union_cnt), _ptr(tok_mask), _ptr(dev_status), _ptr(ws), wsb,
                            _stream(stream))


def pi_sparse_ffn(desc, w, x, batch, idx, cnt, cap, union_idx, union_cnt, tok_mask, y,
                  dev_status, ws, ws_bytes=None, stream=None) -> int:
    return lib().pi_sparse_ffn(ctypes.byref(desc), ctypes.byref(w), _ptr(x), batch, _ptr(idx),
                               _ptr(cnt), cap, _ptr(union_idx), _ptr(union_cnt), _ptr(tok_mask),
                               _ptr(y), _ptr(dev_status), _ptr(ws),
                               ws.numel() if ws_bytes is None else ws_bytes, _stream(stream))


def pi_dense_ffn(desc, w, x, batch, y, ws, ws_bytes=None, stream=None) -> int:
    return lib().pi_dense_ffn(ctypes.byref(desc), ctypes.byref(w), _ptr(x), batch, _ptr(y),
                              _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes,
                              _stream(stream))


def pi_layer_decode(desc, w, x, batch, y, residual, idx_out, cnt_out, dev_status, ws,
                    ws_bytes=None, stream=None) -> int:
    return lib().pi_layer_decode(ctypes.byref(desc), ctypes.byref(w), _ptr(x), batch, _ptr(y),
                                 _ptr(residual), _ptr(idx_out), _ptr(cnt_out), _ptr(dev_status),
                                 _ptr(ws), ws.numel() if ws_bytes is None else ws_bytes,
                                 _stream(stream))


def pi_decode_layers(descs, layers, J, x, chain, y, cnt_out, mask_out, dev_status, ws,
                     ws_bytes=None, stream=None) -> int:
    """descs / layers: lists of R descriptors and weight sets (step j uses
    layer j % R)."""
    R = len(layers)
    if len(descs) != R:
        raise ValueError("one descriptor per layer")
    da = (pi_ffn_desc * R)(*descs)
    wa = (pi_layer_weights * R)(*layers)
    return lib().pi_decode_layers(ctypes.cast(da, ctypes.c_void_p), ctypes.cast(wa, ctypes.c_void_p),
                                  R, J, _ptr(x), chain, _ptr(y), _ptr(cnt_out), _ptr(mask_out),
                                  _ptr(dev_status), _ptr(ws),
                                  ws.numel() if ws_bytes is None else ws_bytes, _stream(stream))


def pi_profile_counts(logits, n, batch, counts, stream=None) -> int:
    return lib().pi_profile_counts(_ptr(logits), n, batch, _ptr(counts), _stream(stream))


def pi_hot_order(counts, n, perm, stream=None) -> int:
    return lib().pi_hot_order(_ptr(counts), n, _ptr(perm), _stream(stream))


def pi_permute_neurons(desc, src, perm, dst, dev_status, stream=None) -> int:
    return lib().pi_permute_neurons(ctypes.byref(desc), ctypes.byref(src), _ptr(perm),
                                    ctypes.byref(dst), _ptr(dev_status), _stream(stream))


def pi_default_cost_model(out: pi_cost_model) -> None:
    lib().pi_default_cost_model(ctypes.byref(out))


def pi_plan_dispatch(desc, batch, p_active, density, allow_dense, model, out) -> int:
    """p_active: None or a host float32 numpy array of n values; model: None
    (the built-in one) or a pi_cost_model; out: a pi_plan filled in place."""
    pa = None
    if p_active is not None:
        import numpy as np
        arr = np.ascontiguousarray(p_active, dtype=np.float32)
        pa = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    return lib().pi_plan_dispatch(ctypes.byref(desc), int(batch), pa, float(density),
                                  int(allow_dense), ctypes.byref(model) if model is not None
                                  else None, ctypes.byref(out))


def pi_pack_weights(desc, W1, W2, packed, stream=None) -> int:
    return lib().pi_pack_weights(ctypes.byref(desc), _ptr(W1), _ptr(W2), _ptr(packed),
                                 _stream(stream))


def pi_layer_decode_static(desc, w, x, y, residual, idx_out, cnt_out, dev_status,
                           stream=None) -> int:
    """pi_layer_decode for one token with the library's fixed scratch instead
    of a workspace (for callers that cannot allocate device memory)."""
    return lib().pi_layer_decode_static(ctypes.byref(desc), ctypes.byref(w), _ptr(x), _ptr(y),
                                        _ptr(residual), _ptr(idx_out), _ptr(cnt_out),
                                        _ptr(dev_status), _stream(stream))


PI_STATIC_SCRATCH_BYTES = 8 << 20


def pi_status_string(status: int) -> str:
    return status_string(status)


def pi_selftest_wait_timeout(dev_status, ws, limit_ns: int, ws_bytes=None, stream=None) -> int:
    return lib().pi_selftest_wait_timeout(_ptr(dev_status), _ptr(ws),
                                          ws.numel() if ws_bytes is None else ws_bytes,
                                          int(limit_ns), _stream(stream))


def pi_selftest_ring_timeout(desc, w, x, idx, cnt, cap, y, dev_status, ws, limit_ns: int,
                             ws_bytes=None, stream=None) -> int:
    return lib().pi_selftest_ring_timeout(ctypes.byref(desc), ctypes.byref(w), _ptr(x), _ptr(idx),
                                          _ptr(cnt), cap, _ptr(y), _ptr(dev_status), _ptr(ws),
                                          ws.numel() if ws_bytes is None else ws_bytes,
                                          int(limit_ns), _stream(stream))


def pi_decode_planned(desc, w, path, x, batch, y, residual, idx_out, cnt_out, dev_status, ws,
                      ws_bytes=None, stream=None) -> int:
    return lib().pi_decode_planned(ctypes.byref(desc), ctypes.byref(w), int(path), _ptr(x), batch,
                                   _ptr(y), _ptr(residual), _ptr(idx_out), _ptr(cnt_out),
                                   _ptr(dev_status), _ptr(ws),
                                   ws.numel() if ws_bytes is None else ws_bytes, _stream(stream))


def pi_decoder_create(desc, w, p_active, density, allow_dense, model, x, y, residual, dev_status,
                      ws, ws_bytes=None):
    """Returns (status, handle); the handle is an opaque int (0 on error).
    p_active: None or a host float32 numpy array of n values."""
    pa = None
    if p_active is not None:
        import numpy as np
        arr = np.ascontiguousarray(p_active, dtype=np.float32)
        pa = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    h = ctypes.c_void_p()
    rc = lib().pi_decoder_create(ctypes.byref(desc), ctypes.byref(w), pa, float(density),
                                 int(allow_dense),
                                 ctypes.byref(model) if model is not None else None, _ptr(x),
                                 _ptr(y), _ptr(residual), _ptr(dev_status), _ptr(ws),
                                 ws.numel() if ws_bytes is None else ws_bytes, ctypes.byref(h))
    return rc, (h.value or 0)


def pi_decoder_run(dec, batch, stream=None) -> int:
    return lib().pi_decoder_run(dec, int(batch), _stream(stream))


def pi_decoder_plan(dec, batch, out) -> int:
    return lib().pi_decoder_plan(dec, int(batch), ctypes.byref(out))


def pi_decoder_destroy(dec) -> None:
    lib().pi_decoder_destroy(dec)


def pi_shard_desc(desc, G, g, out) -> int:
    return lib().pi_shard_desc(ctypes.byref(desc), int(G), int(g), ctypes.byref(out))


def pi_shard_layer(desc, src, G, g, dst, stream=None) -> int:
    return lib().pi_shard_layer(ctypes.byref(desc), ctypes.byref(src), int(G), int(g),
                                ctypes.byref(dst), _stream(stream))


def pi_shard_reduce(parts, G, batch, d, residual, y, stream=None) -> int:
    return lib().pi_shard_reduce(_ptr(parts), int(G), int(batch), int(d), _ptr(residual), _ptr(y),
                                 _stream(stream))
