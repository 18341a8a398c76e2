"""Seeded synthetic workload generator (inputs only).

Thin ctypes binding over ``synth.c``: weight bytes (fp16 / bf16 as uint16),
fp32 biases and fp32 decode-step activations for the activation-sparse
decode FFN.  It contains none of the method's arithmetic; the oracle and the
CUDA library both consume what it writes.  See ``synth.h`` for the recipe.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_HDR = os.path.join(_HERE, "synth.h")
_LIB = os.path.join(_HERE, "libsynth.so")
_GPU_SRC = os.path.join(_HERE, "synth_gpu.cu")
_GPU_LIB = os.path.join(_HERE, "libsynth_gpu.so")
_gpu_lib = None
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1
DTYPES = {"f16": F16, "bf16": BF16}


def build(force: bool = False) -> str:
    """Compile libsynth.so next to the sources (gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def build_gpu(force: bool = False) -> str:
    """Compile libsynth_gpu.so (the generator's CUDA build) next to the sources."""
    stale = (not os.path.exists(_GPU_LIB)) or os.path.getmtime(_GPU_SRC) > os.path.getmtime(_GPU_LIB)
    if force or stale:
        tmp = _GPU_LIB + f".tmp{os.getpid()}"
        cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
               "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _GPU_SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _GPU_LIB)
    return _GPU_LIB


def gpu_lib():
    global _gpu_lib
    with _lock:
        if _gpu_lib is None:
            L = ctypes.CDLL(build_gpu())
            L.sy_gpu_gen_layer.restype = ctypes.c_int
            L.sy_gpu_gen_layer.argtypes = [ctypes.c_int] * 6 + [ctypes.c_uint64, ctypes.c_double] + \
                [ctypes.c_void_p] * 7
            _gpu_lib = L
    return _gpu_lib


class _Spec(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n", ctypes.c_int32), ("r", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("gated", ctypes.c_int32),
                ("layer", ctypes.c_int32), ("seed", ctypes.c_uint64),
                ("alpha", ctypes.c_double), ("zipf_c", ctypes.c_double),
                ("p_cap", ctypes.c_double), ("bias_scale", ctypes.c_double),
                ("noise", ctypes.c_double)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
            L.sy_mix64.restype = u64
            L.sy_mix64.argtypes = [u64]
            L.sy_stream_key.restype = u64
            L.sy_stream_key.argtypes = [u64, ctypes.c_uint32, ctypes.c_uint32]
            L.sy_bits.restype = u64
            L.sy_bits.argtypes = [u64, u64]
            L.sy_uniform.restype = dbl
            L.sy_uniform.argtypes = [u64, u64]
            L.sy_normal.restype = dbl
            L.sy_normal.argtypes = [u64, u64]
            L.sy_round_f16.restype = ctypes.c_uint16
            L.sy_round_f16.argtypes = [dbl]
            L.sy_round_bf16.restype = ctypes.c_uint16
            L.sy_round_bf16.argtypes = [dbl]
            L.sy_probit.restype = dbl
            L.sy_probit.argtypes = [dbl]
            L.sy_relu_m2.restype = dbl
            L.sy_relu_m2.argtypes = [dbl]
            L.sy_zipf_mean.restype = dbl
            L.sy_zipf_mean.argtypes = [i32, dbl, dbl, dbl]
            L.sy_zipf_calibrate.restype = dbl
            L.sy_zipf_calibrate.argtypes = [i32, dbl, dbl, dbl]
            L.sy_zipf_probs.restype = None
            L.sy_zipf_probs.argtypes = [i32, dbl, dbl, dbl, vp]
            L.sy_gen_layer.restype = i32
            L.sy_gen_layer.argtypes = [ctypes.POINTER(_Spec), vp, vp, vp, vp, vp, vp]
            L.sy_gen_x.restype = None
            L.sy_gen_x.argtypes = [u64, i32, i32, i32, vp]
            L.sy_stack_plan.restype = None
            L.sy_stack_plan.argtypes = [u64, i32, i32, dbl, dbl, dbl, dbl, dbl, vp, vp, vp, vp]
            L.sy_num_threads.restype = i32
            L.sy_num_threads.argtypes = []
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- scalars
def stream_key(seed: int, tag: int, layer: int) -> int:
    return lib().sy_stream_key(seed, tag, layer)


def uniform(key: int, k: int) -> float:
    return lib().sy_uniform(key, k)


def normal(key: int, k: int) -> float:
    return lib().sy_normal(key, k)


def round_half(values, dtype: str) -> np.ndarray:
    """Round-to-nearest-even of float64 values to fp16/bf16 bit patterns."""
    f = lib().sy_round_bf16 if DTYPES[dtype] == BF16 else lib().sy_round_f16
    v = np.asarray(values, dtype=np.float64).ravel()
    return np.array([f(float(a)) for a in v], dtype=np.uint16)


def probit(p: float) -> float:
    return lib().sy_probit(p)


def relu_m2(q: float) -> float:
    return lib().sy_relu_m2(q)


def zipf_mean(n: int, alpha: float, c: float, cap: float = 0.9) -> float:
    return lib().sy_zipf_mean(n, alpha, c, cap)


def zipf_calibrate(n: int, alpha: float, target: float, cap: float = 0.9) -> float:
    return lib().sy_zipf_calibrate(n, alpha, target, cap)


def zipf_probs(n: int, alpha: float, c: float, cap: float = 0.9) -> np.ndarray:
    p = np.empty(n, dtype=np.float64)
    lib().sy_zipf_probs(n, alpha, c, cap, _ptr(p))
    return p


def num_threads() -> int:
    return lib().sy_num_threads()


# ---------------------------------------------------------------- tensors
@dataclass
class Layer:
    """One FFN layer's weights as the kernels and the oracle read them."""
    d: int
    n: int
    r: int
    dtype: str                 # "f16" | "bf16"
    gated: bool
    A: np.ndarray              # uint16 [n, r]
    Bm: np.ndarray             # uint16 [r, d]
    b1: np.ndarray             # float32 [n]
    W1: np.ndarray             # uint16 [n, d] or gated [n, 2, d]
    W2: np.ndarray             # uint16 [n, d]
    b2: np.ndarray | None      # float32 [d] or None
    meta: dict = field(default_factory=dict)


def make_layer(d: int, n: int, r: int, dtype: str = "f16", gated: bool = False,
               alpha: float = 0.9, density: float | None = 0.06,
               zipf_c: float | None = None, seed: int = 0, layer: int = 0,
               bias_scale: float = 1.0, noise: float = 0.05, p_cap: float = 0.9,
               with_b2: bool = True) -> Layer:
    """Generate one layer.  Either ``density`` (the Zipf constant is then
    calibrated so that the mean activation probability equals it) or an
    explicit ``zipf_c`` selects the bias profile."""
    if zipf_c is None:
        zipf_c = zipf_calibrate(n, alpha, density, p_cap)
    spec = _Spec(d, n, r, DTYPES[dtype], int(gated), layer, seed, alpha, zipf_c,
                 p_cap, bias_scale, noise)
    A = np.empty((n, r), np.uint16)
    Bm = np.empty((r, d), np.uint16)
    b1 = np.empty(n, np.float32)
    W1 = np.empty((n, 2, d) if gated else (n, d), np.uint16)
    W2 = np.empty((n, d), np.uint16)
    b2 = np.empty(d, np.float32) if with_b2 else None
    rc = lib().sy_gen_layer(ctypes.byref(spec), _ptr(A), _ptr(Bm), _ptr(b1), _ptr(W1),
                            _ptr(W2), _ptr(b2))
    if rc != 0:
        raise RuntimeError(f"sy_gen_layer failed: {rc}")
    meta = dict(alpha=alpha, zipf_c=zipf_c, p_cap=p_cap, bias_scale=bias_scale,
                noise=noise, seed=seed, layer=layer)
    return Layer(d, n, r, dtype, bool(gated), A, Bm, b1, W1, W2, b2, meta)


def gen_x(seed: int, step: int, batch: int, d: int) -> np.ndarray:
    """Decode-step activations x [batch, d] (fp32), fresh per (seed, step)."""
    x = np.empty((batch, d), np.float32)
    lib().sy_gen_x(seed, step, batch, d, _ptr(x))
    return x


def stack_plan(seed: int, L: int, n: int, a_lo: float = 0.7, a_hi: float = 1.2,
               rho_hi: float = 0.15, rho_lo: float = 0.03, cap: float = 0.9):
    """Per-layer (alpha, rho, zipf_c, bias_scale) of a residual stack."""
    out = [np.empty(L, np.float64) for _ in range(4)]
    lib().sy_stack_plan(seed, L, n, a_lo, a_hi, rho_hi, rho_lo, cap, *[_ptr(a) for a in out])
    return tuple(out)


def permute_layer(layer: Layer, perm: np.ndarray) -> Layer:
    """The same layer with its neurons stored in another order: new neuron k
    is old neuron perm[k] (rows of A, b1, W1, W2 move together)."""
    return Layer(layer.d, layer.n, layer.r, layer.dtype, layer.gated,
                 np.ascontiguousarray(layer.A[perm]), layer.Bm,
                 np.ascontiguousarray(layer.b1[perm]),
                 np.ascontiguousarray(layer.W1[perm]),
                 np.ascontiguousarray(layer.W2[perm]), layer.b2,
                 dict(layer.meta, permuted=True))


def make_layer_gpu(d: int, n: int, r: int, dtype: str = "f16", gated: bool = False,
                   alpha: float = 0.9, density: float | None = 0.06,
                   zipf_c: float | None = None, seed: int = 0, layer: int = 0,
                   bias_scale: float = 1.0, noise: float = 0.05, p_cap: float = 0.9,
                   device="cuda", stream=None) -> dict:
    """The same layer as make_layer, generated on the GPU into torch tensors
    (16-bit patterns as int16; b1 / b2 fp32).  For layers too large to build
    quickly on the host."""
    import torch
    if zipf_c is None:
        zipf_c = zipf_calibrate(n, alpha, density, p_cap)
    p = zipf_probs(n, alpha, zipf_c, p_cap)
    b1 = np.array([bias_scale * probit(v) for v in p], dtype=np.float32)
    dev = torch.device(device)
    A = torch.empty((n, r), dtype=torch.int16, device=dev)
    Bm = torch.empty((r, d), dtype=torch.int16, device=dev)
    W1 = torch.empty((n, 2, d) if gated else (n, d), dtype=torch.int16, device=dev)
    W2 = torch.empty((n, d), dtype=torch.int16, device=dev)
    A64 = torch.empty(n * r, dtype=torch.float64, device=dev)
    B64 = torch.empty(r * d, dtype=torch.float64, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream
    rc = gpu_lib().sy_gpu_gen_layer(d, n, r, DTYPES[dtype], int(gated), layer, seed, noise,
                                    A.data_ptr(), Bm.data_ptr(), W1.data_ptr(), W2.data_ptr(),
                                    A64.data_ptr(), B64.data_ptr(), st)
    if rc != 0:
        raise RuntimeError(f"sy_gpu_gen_layer failed: cuda error {rc}")
    del A64, B64
    return dict(d=d, n=n, r=r, dtype=dtype, gated=bool(gated), A=A, Bm=Bm,
                b1=torch.from_numpy(b1).to(dev), W1=W1, W2=W2,
                b2=torch.zeros(d, dtype=torch.float32, device=dev),
                meta=dict(alpha=alpha, zipf_c=zipf_c, p_cap=p_cap, bias_scale=bias_scale,
                          noise=noise, seed=seed, layer=layer))


def to_host_layer(g: dict) -> Layer:
    """Host copy (uint16 patterns) of a GPU-generated layer, for the oracle."""
    cpu = lambda t: t.cpu().numpy()
    return Layer(g["d"], g["n"], g["r"], g["dtype"], g["gated"], cpu(g["A"]).view(np.uint16),
                 cpu(g["Bm"]).view(np.uint16), cpu(g["b1"]), cpu(g["W1"]).view(np.uint16),
                 cpu(g["W2"]).view(np.uint16), cpu(g["b2"]), dict(g["meta"]))
