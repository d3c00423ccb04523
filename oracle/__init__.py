"""fp64 CPU oracle for exact softmax attention and its gradients.

TEST INFRASTRUCTURE ONLY.  This package is the yardstick that the CUDA
library is checked against: only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it.  It shares no code with the CUDA
path and never calls it; the CUDA path never calls it either.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, the
textbook definition of softmax attention and its analytic gradient written
out row by row).  This module compiles that file with gcc and wraps it with
ctypes.  Every function takes and returns numpy arrays in the layout
[B, H, N, d] (L and D: [B, H, N]); inputs of any float type are converted
exactly to float64 first.

Source of the method: "Training Transformers and Hybrid models on AMD
Instinct MI300X Accelerators", section "Flash Attention" (the
FlashAttention-2 forward and backward, with the forward's activations
recomputed in the backward), and section "Harnessing the MI300 Hardware
Specs".  The pages print no formula; the definition used is the textbook one
stated at the top of ``attn_oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libattn_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle shared library with gcc (OpenMP when available).

    Returns the path of the built library.  No -ffast-math: the oracle keeps
    IEEE double semantics.
    """
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its ABI."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib_path = path or build()
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lp = ctypes.POINTER(ctypes.c_long)
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, L, L, L, ctypes.c_int, L, lp,
                                        ctypes.c_double, dp, dp, ctypes.c_int]
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_fwd_bwd.argtypes = [dp, dp, dp, dp, L, L, L, ctypes.c_int, L, lp,
                                            ctypes.c_double, dp, dp, dp, dp, dp,
                                            dp, ctypes.c_int]
        lib.oracle_attn_fwd_bwd.restype = ctypes.c_int
        lib.oracle_attn_head_rows.argtypes = [dp, dp, dp, dp, L, L, ctypes.c_int, L, lp,
                                              ctypes.c_double, L, lp, L, lp, dp, dp, dp,
                                              dp, dp, ctypes.c_int]
        lib.oracle_attn_head_rows.restype = ctypes.c_int
        lib.oracle_attn_bwd_budget.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, ctypes.c_int,
                                               ctypes.c_double, dp, dp, dp, dp, dp,
                                               ctypes.c_int]
        lib.oracle_attn_bwd_budget.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    """Exact conversion to a C-contiguous float64 array (torch or numpy)."""
    if hasattr(x, "detach"):  # torch tensor, possibly bf16
        x = x.detach().to("cpu")
        import torch  # local: the oracle itself does not need torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _doc_map(doc, heads_per_batch: int, rows: int):
    """A document map [B, N] (first position of each position's document),
    repeated for every head: [B*H, N] C longs, or None."""
    if doc is None:
        return None, None
    if hasattr(doc, "detach"):
        doc = doc.detach().to("cpu").numpy()
    a = np.asarray(doc, dtype=np.int64)
    if a.ndim == 1:
        a = a[None, :]
    if a.shape[-1] != rows:
        raise ValueError("document map must have N = %d columns" % rows)
    a = np.ascontiguousarray(np.repeat(a, heads_per_batch, axis=0).astype(np.dtype("l")))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_long))


def max_threads(lib=None) -> int:
    return int((lib or load()).oracle_max_threads())


def attention_forward(q, k, v, causal: bool, scale: float, threads: int = 0, lib=None,
                      window: int = 0, doc=None):
    """O [B,H,N,d] and L [B,H,N] (natural-log log-sum-exp), both float64.

    window > 0 (causal only): query i sees keys i - window < j <= i.
    doc [B, N] (causal only): query i sees keys from doc[b, i] on, the first
    position of its document."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share the shape [B, H, N, d]")
    B, H, N, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, N), dtype=np.float64)
    doc_a, doc_p = _doc_map(doc, H, N)
    st = (lib or load()).oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B * H, N, d,
                                         int(bool(causal)), int(window), doc_p, float(scale),
                                         _ptr(o),
                                         _ptr(lse), int(threads))
    if st != 0:
        raise RuntimeError("oracle_attn_fwd failed with status %d" % st)
    return o, lse


def attention_forward_backward(q, k, v, do, causal: bool, scale: float,
                               threads: int = 0, lib=None, window: int = 0, doc=None) -> dict:
    """Exact forward and analytic backward in float64.

    Returns a dict with O, L, D (= rowsum(dO * O)), dQ, dK, dV.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if q.ndim != 4 or any(t.shape != q.shape for t in (k, v, do)):
        raise ValueError("q, k, v, do must share the shape [B, H, N, d]")
    B, H, N, d = q.shape
    out = {name: np.zeros_like(q) for name in ("O", "dQ", "dK", "dV")}
    out["L"] = np.zeros((B, H, N), dtype=np.float64)
    out["D"] = np.zeros((B, H, N), dtype=np.float64)
    doc_a, doc_p = _doc_map(doc, H, N)
    st = (lib or load()).oracle_attn_fwd_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(do), B * H, N, d, int(bool(causal)), int(window),
        doc_p, float(scale), _ptr(out["O"]), _ptr(out["L"]), _ptr(out["D"]),
        _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]), int(threads))
    if st != 0:
        raise RuntimeError("oracle_attn_fwd_bwd failed with status %d" % st)
    return out


def attention_head_rows(q, k, v, do, causal: bool, scale: float, q_rows, k_rows,
                        threads: int = 0, lib=None, window: int = 0, doc=None) -> dict:
    """Sampled rows of one head ([N, d] inputs), for shapes too large to do in full.

    Returns O, L, dQ at the query rows ``q_rows`` and dK, dV at the key rows
    ``k_rows`` (float64).  The forward statistics of every row are computed,
    because dK_j and dV_j depend on L_i and D_i of all query rows.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if q.ndim != 2 or any(t.shape != q.shape for t in (k, v, do)):
        raise ValueError("q, k, v, do must share the shape [N, d]")
    N, d = q.shape
    qr = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int64)).astype(np.dtype("l"))
    kr = np.ascontiguousarray(np.asarray(k_rows, dtype=np.int64)).astype(np.dtype("l"))
    out = {"O": np.zeros((len(qr), d)), "L": np.zeros(len(qr)), "dQ": np.zeros((len(qr), d)),
           "dK": np.zeros((len(kr), d)), "dV": np.zeros((len(kr), d))}
    lp = ctypes.POINTER(ctypes.c_long)
    doc_a, doc_p = _doc_map(doc, 1, N)  # one head: doc is [N]
    st = (lib or load()).oracle_attn_head_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(do), N, d, int(bool(causal)), int(window), doc_p,
        float(scale),
        len(qr), qr.ctypes.data_as(lp), len(kr), kr.ctypes.data_as(lp), _ptr(out["O"]),
        _ptr(out["L"]), _ptr(out["dQ"]), _ptr(out["dK"]), _ptr(out["dV"]), int(threads))
    if st != 0:
        raise RuntimeError("oracle_attn_head_rows failed with status %d" % st)
    return out


def backward_rounding_budget(q, k, v, do, causal: bool, scale: float, L, D, threads: int = 0,
                             lib=None) -> dict:
    """The sums that bound the rounding of P and dS to 8 bits in a backward
    pass (plain masks), from the forward statistics L, D of
    ``attention_forward_backward``: vP[j] = sum_i P_ij^2 dO_i^2,
    vK[j] = sum_i dS_ij^2 q_i^2, vQ[i] = sum_j dS_ij^2 k_j^2 (elementwise over
    the head dim, [B,H,N,d]), nvis[j] = the query rows that see key j
    ([B,H,N]), and dsmax = max |dS| per head ([B,H])."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    L, D = _f64(L), _f64(D)
    B, H, N, d = q.shape
    out = {name: np.zeros_like(q) for name in ("vP", "vK", "vQ")}
    out["nvis"] = np.zeros((B, H, N))
    out["dsmax"] = np.zeros((B, H))
    st = (lib or load()).oracle_attn_bwd_budget(
        _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(L), _ptr(D), B * H, N, d, int(bool(causal)),
        float(scale), _ptr(out["vP"]), _ptr(out["vK"]), _ptr(out["vQ"]), _ptr(out["nvis"]),
        _ptr(out["dsmax"]), int(threads))
    if st != 0:
        raise RuntimeError("oracle_attn_bwd_budget failed with status %d" % st)
    return out
