"""fp64 CPU oracle for the Mamba-2 state-space layer and its backward pass.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the test suite,
the smoke check and the benchmark's CPU-baseline leg may import it.  It shares
no code with the CUDA path and never calls it.

The arithmetic is in ``ssd_oracle.c`` (the recurrence and its adjoint written
out step by step; the formulas are at the top of that file).  This module
compiles it with gcc and wraps it with ctypes.  Layouts: x, dy, y, dx
[Bt, T, H, P]; dt, ddt [Bt, T, H]; A, D, dA, dD [H]; B, C, dB, dC
[Bt, T, G, N].  Inputs of any float type are converted exactly to float64.

Source: "Training Transformers and Hybrid models on AMD Instinct MI300X
Accelerators", section "Mamba-2" (the backward kernel of the hybrid model's
state-space layer, by a prefix scan and a reverse scan).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libssd_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the SSD oracle with gcc (OpenMP when available), IEEE doubles."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True,
                       text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        dp = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.oracle_ssd_fwd.argtypes = [dp] * 6 + [L] * 6 + [dp, ctypes.c_int]
        lib.oracle_ssd_fwd.restype = ctypes.c_int
        lib.oracle_ssd_fwd_bwd.argtypes = [dp] * 7 + [L] * 6 + [dp] * 7 + [ctypes.c_int]
        lib.oracle_ssd_fwd_bwd.restype = ctypes.c_int
        lib.oracle_ssd_max_threads.argtypes = []
        lib.oracle_ssd_max_threads.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch

        a = a.detach().to("cpu").to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(x, dt, A, B, C, D):
    if x.ndim != 4 or B.ndim != 4 or C.shape != B.shape:
        raise ValueError("x must be [Bt, T, H, P]; B and C [Bt, T, G, N]")
    Bt, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if B.shape[:2] != (Bt, T) or dt.shape != (Bt, T, H) or A.shape != (H,) or D.shape != (H,):
        raise ValueError("inconsistent shapes")
    if G == 0 or H % G:
        raise ValueError("heads must split evenly into groups")
    return Bt, T, H, G, N, P


def max_threads(lib=None) -> int:
    return int((lib or load()).oracle_ssd_max_threads())


def ssd_forward(x, dt, A, B, C, D, threads: int = 0, lib=None) -> np.ndarray:
    """y [Bt, T, H, P] in float64."""
    x, dt, A, B, C, D = (_f64(t) for t in (x, dt, A, B, C, D))
    Bt, T, H, G, N, P = _shapes(x, dt, A, B, C, D)
    y = np.zeros_like(x)
    st = (lib or load()).oracle_ssd_fwd(_p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), Bt, T, H, G,
                                        N, P, _p(y), int(threads))
    if st:
        raise RuntimeError("oracle_ssd_fwd failed with status %d" % st)
    return y


def ssd_forward_backward(x, dt, A, B, C, D, dy, threads: int = 0, lib=None) -> dict:
    """y and the gradients of <dy, y>: dx, ddt, dA, dB, dC, dD (float64)."""
    x, dt, A, B, C, D, dy = (_f64(t) for t in (x, dt, A, B, C, D, dy))
    Bt, T, H, G, N, P = _shapes(x, dt, A, B, C, D)
    if dy.shape != x.shape:
        raise ValueError("dy must match x")
    out = {"y": np.zeros_like(x), "dx": np.zeros_like(x), "ddt": np.zeros_like(dt),
           "dA": np.zeros_like(A), "dB": np.zeros_like(B), "dC": np.zeros_like(C),
           "dD": np.zeros_like(D)}
    st = (lib or load()).oracle_ssd_fwd_bwd(
        _p(x), _p(dt), _p(A), _p(B), _p(C), _p(D), _p(dy), Bt, T, H, G, N, P, _p(out["y"]),
        _p(out["dx"]), _p(out["ddt"]), _p(out["dA"]), _p(out["dB"]), _p(out["dC"]),
        _p(out["dD"]), int(threads))
    if st:
        raise RuntimeError("oracle_ssd_fwd_bwd failed with status %d" % st)
    return out
