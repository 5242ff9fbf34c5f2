"""fp64 CPU oracle for grouped-convolution backward-weight.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``, never by the product package.  It shares no
code with the CUDA path.

The C file ``wgrad_oracle.c`` holds the arithmetic (direct loops over the
definitions of the weight gradient, the forward convolution and the
backward-data gradient, see its header).  This module compiles it
with gcc + OpenMP into ``oracle/_lib/liboracle.so`` and wraps it for numpy.

A problem is a dict with keys ``ndim`` (1, 2 or 3), ``G``, ``N``, ``C``, ``K``
(channels per group) and the per-dimension lists ``in``, ``filt``, ``stride``,
``dil``, ``pad_l``, ``pad_r`` of length ``ndim``, outermost spatial dim first.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wgrad_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _OProblem(ctypes.Structure):
    _fields_ = [("G", ctypes.c_int), ("N", ctypes.c_int), ("C", ctypes.c_int), ("K", ctypes.c_int),
                ("in_", ctypes.c_int * 3), ("filt", ctypes.c_int * 3), ("stride", ctypes.c_int * 3),
                ("dil", ctypes.c_int * 3), ("pad_l", ctypes.c_int * 3), ("pad_r", ctypes.c_int * 3)]


def build(force: bool = False) -> str:
    """Compile the oracle library (gcc -O2 -fopenmp).  Returns its path."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            os.makedirs(_LIBDIR, exist_ok=True)
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.orc_out_len.restype = ctypes.c_int
        lib.orc_out_len.argtypes = [ctypes.c_int] * 6
        lib.orc_threads.restype = ctypes.c_int
        lib.orc_decode16.argtypes = [ctypes.c_void_p, ctypes.c_long, ctypes.c_int, dp]
        lib.orc_wgrad.argtypes = [ctypes.POINTER(_OProblem), dp, dp, dp, dp]
        lib.orc_wgrad_at.argtypes = [ctypes.POINTER(_OProblem), dp, dp, ctypes.c_void_p, ctypes.c_long,
                                     dp, dp]
        lib.orc_conv_fwd.argtypes = [ctypes.POINTER(_OProblem), dp, dp, dp]
        lib.orc_dgrad.argtypes = [ctypes.POINTER(_OProblem), dp, dp, dp, dp]
        _lib = lib
    return _lib


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _spatial3(p: dict, key: str, fill: int) -> list:
    v = list(p[key])
    if len(v) != p["ndim"]:
        raise ValueError(f"{key} must have {p['ndim']} entries")
    return [fill] * (3 - len(v)) + v


def _struct(p: dict) -> _OProblem:
    s = _OProblem()
    s.G, s.N, s.C, s.K = p["G"], p["N"], p["C"], p["K"]
    for name, field, fill in (("in", "in_", 1), ("filt", "filt", 1), ("stride", "stride", 1),
                              ("dil", "dil", 1), ("pad_l", "pad_l", 0), ("pad_r", "pad_r", 0)):
        getattr(s, field)[:] = _spatial3(p, name, fill)
    return s


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return _load().orc_threads()


def out_dims(p: dict) -> list:
    """Output spatial lengths (ndim entries) by the standard convolution rule."""
    lib = _load()
    return [lib.orc_out_len(p["in"][i], p["filt"][i], p["stride"][i], p["dil"][i], p["pad_l"][i],
                            p["pad_r"][i]) for i in range(p["ndim"])]


def shapes(p: dict) -> dict:
    """Element shapes of X (N,*in,G,C), dY (N,*out,G,K) and dW (G,K,*filt,C)."""
    o = out_dims(p)
    return {"x": (p["N"], *p["in"], p["G"], p["C"]),
            "dy": (p["N"], *o, p["G"], p["K"]),
            "dw": (p["G"], p["K"], *p["filt"], p["C"])}


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of bf16/fp16 words."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().orc_decode16(b.ctypes.data, b.size, 1 if dtype == "bf16" else 0, _dp(out))
    return out


def wgrad(p: dict, x: np.ndarray, dy: np.ndarray):
    """Full dW and A = sum |dY*X| (float64, shape G,K,*filt,C)."""
    sh = shapes(p)
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(sh["x"])
    dy = np.ascontiguousarray(dy, dtype=np.float64).reshape(sh["dy"])
    dw = np.empty(sh["dw"], dtype=np.float64)
    ab = np.empty(sh["dw"], dtype=np.float64)
    _load().orc_wgrad(ctypes.byref(_struct(p)), _dp(x), _dp(dy), _dp(dw), _dp(ab))
    return dw, ab


def wgrad_at(p: dict, x: np.ndarray, dy: np.ndarray, flat_idx: np.ndarray):
    """dW and A at the given flat indices of the G,K,*filt,C tensor."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    dy = np.ascontiguousarray(dy, dtype=np.float64)
    idx = np.ascontiguousarray(flat_idx, dtype=np.int64)
    out = np.empty(idx.shape, dtype=np.float64)
    ab = np.empty(idx.shape, dtype=np.float64)
    _load().orc_wgrad_at(ctypes.byref(_struct(p)), _dp(x), _dp(dy), idx.ctypes.data, idx.size, _dp(out),
                         _dp(ab))
    return out, ab


def conv_fwd(p: dict, x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Forward grouped convolution y (N,*out,G,K) of X with weights w (G,K,*filt,C)."""
    sh = shapes(p)
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(sh["x"])
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(sh["dw"])
    y = np.empty(sh["dy"], dtype=np.float64)
    _load().orc_conv_fwd(ctypes.byref(_struct(p)), _dp(x), _dp(w), _dp(y))
    return y


def dgrad(p: dict, dy: np.ndarray, w: np.ndarray):
    """Backward-data: dX (N,*in,G,C) from dY (N,*out,G,K) and W (G,K,*filt,C), and
    A = sum |dY*W| over the same terms (float64)."""
    sh = shapes(p)
    dy = np.ascontiguousarray(dy, dtype=np.float64).reshape(sh["dy"])
    w = np.ascontiguousarray(w, dtype=np.float64).reshape(sh["dw"])
    dx = np.empty(sh["x"], dtype=np.float64)
    ab = np.empty(sh["x"], dtype=np.float64)
    _load().orc_dgrad(ctypes.byref(_struct(p)), _dp(dy), _dp(w), _dp(dx), _dp(ab))
    return dx, ab
