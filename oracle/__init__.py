"""CPU FP64 oracle for the DDPM core -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

The arithmetic lives in ``ddpm_oracle.c`` (plain C loops, FP64, OpenMP over
independent outputs).  This module builds it with gcc on first use and wraps
it with ctypes, taking and returning numpy float64 arrays.

Source of the method: "lartpang/DynamicConvolutionOperator" README (the
Dynamic Dilated Pyramid Module of HDFNet, ECCV 2020), sections "问题与目标",
"CUDA 动态过滤", "CUDA 融合生成器推理" and "CUDA Flash 式融合训练".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddpm_oracle.c")
_HDR = os.path.join(_HERE, "ddpm_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libddpm_oracle.so")
_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("C", ctypes.c_int), ("H", ctypes.c_int),
                ("W", ctypes.c_int), ("K", ctypes.c_int), ("dil", ctypes.c_int * 3),
                ("bf16", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compile ddpm_oracle.c into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            d = P(ctypes.c_double)
            sp = P(_Shape)
            i64p = P(ctypes.c_int64)
            lib.ddpmo_round_bf16.argtypes = [ctypes.c_double]
            lib.ddpmo_round_bf16.restype = ctypes.c_double
            lib.ddpmo_tap.argtypes = [sp, d, d, d, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.ddpmo_tap.restype = ctypes.c_double
            lib.ddpmo_generate_taps.argtypes = [sp, d, d, d, d]
            lib.ddpmo_forward.argtypes = [sp, d, d, d, d, d]
            lib.ddpmo_filter.argtypes = [sp, d, d, d]
            lib.ddpmo_forward_points.argtypes = [sp, d, d, d, d, ctypes.c_int64, i64p, d]
            lib.ddpmo_filter_points.argtypes = [sp, d, d, ctypes.c_int64, i64p, d]
            lib.ddpmo_backward.argtypes = [sp, d, d, d, d, d, d, d, d, d]
            lib.ddpmo_backward_points.argtypes = [sp, d, d, d, d, d, ctypes.c_int, ctypes.c_int64, i64p, d]
            lib.ddpmo_filter_backward.argtypes = [sp, d, d, d, d, d]
            lib.ddpmo_num_threads.argtypes = []
            for f in ("ddpmo_generate_taps", "ddpmo_forward", "ddpmo_filter", "ddpmo_forward_points",
                      "ddpmo_filter_points", "ddpmo_backward", "ddpmo_backward_points", "ddpmo_filter_backward",
                      "ddpmo_num_threads"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(B, C, H, W, K, dilations, bf16):
    s = _Shape()
    s.B, s.C, s.H, s.W, s.K = int(B), int(C), int(H), int(W), int(K)
    for i in range(3):
        s.dil[i] = int(dilations[i])
    s.bf16 = 1 if bf16 else 0
    return s


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _idx(idx):
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    return idx, idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def num_threads() -> int:
    """OpenMP threads the oracle uses (honours OMP_NUM_THREADS)."""
    return int(_load().ddpmo_num_threads())


def round_bf16(v: float) -> float:
    """Round one value to the nearest bfloat16 (ties to even)."""
    return float(_load().ddpmo_round_bf16(float(v)))


def tap(y, Wg, bias, K, dilations, b, o, h, w, bf16=False) -> float:
    """One generator output T[b,o,h,w] = bias[o] + sum_j Wg[o,j] y[b,j,h,w]."""
    y, Wg = _f64(y), _f64(Wg)
    bias = None if bias is None else _f64(bias)
    B, C, H, W = y.shape
    s = _shape(B, C, H, W, K, dilations, bf16)
    return float(_load().ddpmo_tap(ctypes.byref(s), _ptr(y), _ptr(Wg), _ptr(bias), b, o, h, w))


def generate_taps(y, Wg, bias, K, dilations=(1, 3, 5), bf16=False) -> np.ndarray:
    """Materialised taps T [B, 3*C*K*K, H, W]."""
    y, Wg = _f64(y), _f64(Wg)
    bias = None if bias is None else _f64(bias)
    B, C, H, W = y.shape
    s = _shape(B, C, H, W, K, dilations, bf16)
    T = np.empty((B, 3 * C * K * K, H, W), dtype=np.float64)
    _check(_load().ddpmo_generate_taps(ctypes.byref(s), _ptr(y), _ptr(Wg), _ptr(bias), _ptr(T)), "generate_taps")
    return T


def forward(x, y, Wg, bias, K, dilations=(1, 3, 5), bf16=False) -> np.ndarray:
    """Fused generator + dynamic dilated depthwise filter: out [B, 4C, H, W]."""
    x, y, Wg = _f64(x), _f64(y), _f64(Wg)
    bias = None if bias is None else _f64(bias)
    B, C, H, W = x.shape
    s = _shape(B, C, H, W, K, dilations, bf16)
    out = np.empty((B, 4 * C, H, W), dtype=np.float64)
    _check(_load().ddpmo_forward(ctypes.byref(s), _ptr(x), _ptr(y), _ptr(Wg), _ptr(bias), _ptr(out)), "forward")
    return out


def filter_pregenerated(x, T, K, dilations=(1, 3, 5)) -> np.ndarray:
    """Dynamic filter with taps given: out [B, 4C, H, W]."""
    x, T = _f64(x), _f64(T)
    B, C, H, W = x.shape
    s = _shape(B, C, H, W, K, dilations, False)
    out = np.empty((B, 4 * C, H, W), dtype=np.float64)
    _check(_load().ddpmo_filter(ctypes.byref(s), _ptr(x), _ptr(T), _ptr(out)), "filter")
    return out


def forward_points(x, y, Wg, bias, K, idx, dilations=(1, 3, 5), bf16=False) -> np.ndarray:
    """out.flat[idx] of the fused forward, without computing the rest."""
    x, y, Wg = _f64(x), _f64(y), _f64(Wg)
    bias = None if bias is None else _f64(bias)
    B, C, H, W = x.shape
    s = _shape(B, C, H, W, K, dilations, bf16)
    idx, ip = _idx(idx)
    vals = np.empty(idx.shape[0], dtype=np.float64)
    _check(_load().ddpmo_forward_points(ctypes.byref(s), _ptr(x), _ptr(y), _ptr(Wg), _ptr(bias),
                                        idx.shape[0], ip, _ptr(vals)), "forward_points")
    return vals


def filter_points(x, T, K, idx, dilations=(1, 3, 5)) -> np.ndarray:
    """out.flat[idx] of the filter with given taps."""
    x, T = _f64(x), _f64(T)
    B, C, H, W = x.shape
    s = _shape(B, C, H, W, K, dilations, False)
    idx, ip = _idx(idx)
    vals = np.empty(idx.shape[0], dtype=np.float64)
    _check(_load().ddpmo_filter_points(ctypes.byref(s), _ptr(x), _ptr(T), idx.shape[0], ip, _ptr(vals)),
           "filter_points")
    return vals


def backward(g, x, y, Wg, bias, K, dilations=(1, 3, 5), bf16=False):
    """Gradients of L = <g, out>: returns (dx, dy, dW, dbias)."""
    g, x, y, Wg = _f64(g), _f64(x), _f64(y), _f64(Wg)
    bias = None if bias is None else _f64(bias)
    B, C, H, W = x.shape
    O = 3 * C * K * K
    s = _shape(B, C, H, W, K, dilations, bf16)
    dx = np.empty((B, C, H, W))
    dy = np.empty((B, C, H, W))
    dW = np.empty((O, C))
    db = np.empty((O,))
    _check(_load().ddpmo_backward(ctypes.byref(s), _ptr(g), _ptr(x), _ptr(y), _ptr(Wg), _ptr(bias),
                                  _ptr(dx), _ptr(dy), _ptr(dW), _ptr(db)), "backward")
    return dx, dy, dW, db


def filter_backward(g, x, T, K, dilations=(1, 3, 5)):
    """Gradients of L = <g, filter_pregenerated(x, T)> (README section "CUDA 动态过滤":
    the backward of the filter with given taps forms dX and dK without a patch
    matrix): returns (dx [B,C,H,W], dT [B,O,H,W])."""
    g, x, T = _f64(g), _f64(x), _f64(T)
    B, C, H, W = x.shape
    s = _shape(B, C, H, W, K, dilations, False)
    dx = np.empty((B, C, H, W))
    dT = np.empty_like(T)
    _check(_load().ddpmo_filter_backward(ctypes.byref(s), _ptr(g), _ptr(x), _ptr(T), _ptr(dx), _ptr(dT)),
           "filter_backward")
    return dx, dT


_WHICH = {"dx": 0, "dy": 1, "dW": 2, "dbias": 3}


def backward_points(g, x, y, Wg, bias, K, which, idx, dilations=(1, 3, 5), bf16=False) -> np.ndarray:
    """One gradient tensor ('dx', 'dy', 'dW' or 'dbias') at flat indices idx."""
    g, x, y, Wg = _f64(g), _f64(x), _f64(y), _f64(Wg)
    bias = None if bias is None else _f64(bias)
    B, C, H, W = x.shape
    s = _shape(B, C, H, W, K, dilations, bf16)
    idx, ip = _idx(idx)
    vals = np.empty(idx.shape[0], dtype=np.float64)
    _check(_load().ddpmo_backward_points(ctypes.byref(s), _ptr(g), _ptr(x), _ptr(y), _ptr(Wg), _ptr(bias),
                                         _WHICH[which], idx.shape[0], ip, _ptr(vals)), "backward_points")
    return vals
