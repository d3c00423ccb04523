"""ctypes binding of the C ABI in ``include/attn.h``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libattn_gb300.so``.  PyTorch supplies device memory (outputs and
the backward's workspace are allocated here with ``torch.empty`` unless the
caller passes them) and the current CUDA stream.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_WORKSPACE = 5
ATTN_ERR_DEVICE = 6
ATTN_ERR_TOO_LARGE = 7

# How attn_bwd forms dQ (attn_dq_method_t in include/attn.h).
ATTN_DQ_AUTO = 0
ATTN_DQ_REDUCE = 1
ATTN_DQ_SEPARATE = 2

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, fn: str, status: int, text: str):
        super().__init__("%s failed: %s (status %d)" % (fn, text, status))
        self.status = status


def load_library(path: str | None = None):
    """Load ``libattn_gb300.so`` (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                "CUDA library %s is not built; run __graft_entry__.build() (needs nvcc). "
                "There is no CPU fallback." % p)
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "attn_fwd": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]),
            "attn_fwd_ex": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, f, vp]),
            "attn_fwd_fp8": (i, [vp, vp, vp, f, f, f, vp, vp, i, i, i, i, i, f, vp]),
            "attn_bwd_workspace_size": (sz, [i, i, i, i]),
            "attn_bwd": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]),
            "attn_bwd_ex": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, f, vp,
                                sz, vp]),
            "attn_bwd_fp8": (i, [vp, vp, vp, vp, vp, vp, f, f, f, f, f, vp, vp, vp, vp, i, i, i,
                                 i, i, f, vp, sz, vp]),
            "attn_bwd_opts": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, f,
                                  i, vp, sz, vp]),
            "attn_bwd_main_dkdv": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]),
            "attn_bwd_dq": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]),
            "attn_bwd_preprocess": (i, [vp, vp, vp, i, i, i, i, vp, sz, vp]),
            "attn_bwd_main": (i, [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]),
            "attn_bwd_dq_convert": (i, [vp, i, i, i, i, f, vp, sz, vp]),
            "attn_bwd_noalloc": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]),
            "ssd_workspace_size": (sz, [i, i, i, i, i, i]),
            "ssd_fwd": (i, [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]),
            "ssd_bwd": (i, [vp] * 13 + [i, i, i, i, i, i, vp, sz, vp]),
            "attn_last_device_error": (i, [vp]),
            "attn_device_error_word": (i, [vp, ctypes.POINTER(ctypes.c_int)]),
            "attn_watchdog_selftest": (i, [ctypes.c_uint64, vp]),
            "attn_status_string": (ctypes.c_char_p, [i]),
            "attn_version": (i, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != ATTN_OK:
        raise AttnError(fn, status, status_string(status))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _shape4(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError("%s must be [B, H, N, d], got %s" % (name, tuple(t.shape)))
    return tuple(t.shape)


def _check_tensor(t: torch.Tensor, name: str, shape, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _doc_ptr(doc, B: int, N: int):
    """Device pointer of a document map (int32 CUDA tensor [B, N], contiguous), or None."""
    if doc is None:
        return None
    _check_tensor(doc, "doc", (B, N), torch.int32)
    return doc.data_ptr()


def _default_scale(d: int, scale):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_bwd_workspace_size(B, H, N, d))


def alloc_workspace(B: int, H: int, N: int, d: int, device) -> torch.Tensor:
    """A uint8 device buffer of the size attn_bwd needs (torch allocations are
    256-byte aligned)."""
    n = max(attn_bwd_workspace_size(B, H, N, d), 256)
    return torch.empty(n, dtype=torch.uint8, device=device)


def attn_fwd(q, k, v, causal: bool, scale=None, out=None, lse=None, stream=None, window=0,
             doc=None):
    """O = softmax(scale q k^T [+ causal mask]) v and the row log-sum-exp L.

    q, k, v: bf16 CUDA tensors [B, H, N, d] (d = 64 or 128), contiguous.
    window > 0 (causal only): query i sees keys i - window < j <= i.
    doc (causal only): int32 CUDA tensor [B, N], the first position of each
    position's document; query i sees keys doc[b, i] <= j <= i.
    Returns (O bf16 [B, H, N, d], L fp32 [B, H, N]).
    """
    B, H, N, d = _shape4(q, "q")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_tensor(t, n, (B, H, N, d))
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(out, "out", (B, H, N, d))
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    st = load_library().attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, H, N, d, int(bool(causal)), int(window),
                                    _doc_ptr(doc, B, N), _default_scale(d, scale),
                                    _stream(stream))
    _check("attn_fwd_ex", st)
    return out, lse


def _check_fp8(t: torch.Tensor, name: str, shape):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.element_size() != 1 or t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError("%s must hold e4m3 bytes (float8_e4m3fn or uint8), got %s"
                         % (name, t.dtype))
    if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError("%s must be contiguous with shape %s" % (name, tuple(shape)))


def attn_fwd_fp8(q8, k8, v8, descales, causal: bool, scale=None, out=None, lse=None,
                 stream=None):
    """O (bf16) and L (fp32) of exact attention over e4m3 inputs.

    q8, k8, v8: e4m3 bytes [B, H, N, 128] (float8_e4m3fn or uint8 views);
    descales: (q_descale, k_descale, v_descale), the factors that turn the
    stored values into the values they stand for.
    """
    B, H, N, d = _shape4(q8, "q8")
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _check_fp8(t, n, (B, H, N, d))
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None \
        else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _check_tensor(out, "out", (B, H, N, d))
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    qd, kd, vd = (float(x) for x in descales)
    st = load_library().attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), qd, kd, vd,
                                     out.data_ptr(), lse.data_ptr(), B, H, N, d,
                                     int(bool(causal)), _default_scale(d, scale),
                                     _stream(stream))
    _check("attn_fwd_fp8", st)
    return out, lse


def attn_bwd_fp8(q8, k8, v8, o, do8, lse, descales, ds_scale: float, causal: bool, scale=None,
                 ds_amax=None, workspace=None, stream=None):
    """dQ, dK, dV (bf16) of exact attention with e4m3 operands.

    q8, k8, v8, do8: e4m3 bytes [B, H, N, 128]; descales: (q, k, v, dO)
    factors; o (bf16) and lse: the forward's outputs; ds_scale: the factor
    dS is multiplied by before its rounding to e4m3 (keep ds_scale x
    max|dS| <= 448).  ds_amax: a 1-element float32 CUDA tensor that receives
    the largest |dS| of the call (or None).  Returns (dQ, dK, dV).
    """
    B, H, N, d = _shape4(q8, "q8")
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8"), (do8, "do8")):
        _check_fp8(t, n, (B, H, N, d))
    _check_tensor(o, "o", (B, H, N, d))
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    if ds_amax is not None:
        _check_tensor(ds_amax, "ds_amax", (1,), torch.float32)
    dq, dk, dv = (torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
                  for _ in range(3))
    if workspace is None:
        workspace = alloc_workspace(B, H, N, d, q8.device)
    qd, kd, vd, dod = (float(x) for x in descales)
    st = load_library().attn_bwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(),
                                     do8.data_ptr(), lse.data_ptr(), qd, kd, vd, dod,
                                     float(ds_scale), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr(),
                                     None if ds_amax is None else ds_amax.data_ptr(), B, H, N,
                                     d, int(bool(causal)), _default_scale(d, scale),
                                     workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    _check("attn_bwd_fp8", st)
    return dq, dk, dv


def attn_bwd(q, k, v, o, do, lse, causal: bool, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None, window=0, doc=None, dq_method=ATTN_DQ_AUTO):
    """dQ, dK, dV of exact attention (the fused backward).

    o, lse: the forward's outputs; do: the upstream gradient of o.
    dq_method: ATTN_DQ_AUTO, ATTN_DQ_REDUCE (the main kernel reduces dQ
    partials into an fp32 accumulator) or ATTN_DQ_SEPARATE (a separate
    query-stationary dQ pass).
    Returns (dQ, dK, dV), bf16 [B, H, N, d].
    """
    B, H, N, d = _shape4(q, "q")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check_tensor(t, n, (B, H, N, d))
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check_tensor(t, n, (B, H, N, d))
    if workspace is None:
        workspace = alloc_workspace(B, H, N, d, q.device)
    st = load_library().attn_bwd_opts(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                      dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                      int(bool(causal)), int(window), _doc_ptr(doc, B, N),
                                      _default_scale(d, scale), int(dq_method),
                                      workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(stream))
    _check("attn_bwd_opts", st)
    return dq, dk, dv


def attn_bwd_preprocess(o, do, lse, workspace, stream=None):
    B, H, N, d = _shape4(o, "o")
    st = load_library().attn_bwd_preprocess(o.data_ptr(), do.data_ptr(), lse.data_ptr(), B, H, N,
                                            d, workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream))
    _check("attn_bwd_preprocess", st)


def attn_bwd_main(q, k, v, do, dk, dv, causal: bool, workspace, scale=None, stream=None):
    B, H, N, d = _shape4(q, "q")
    st = load_library().attn_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                      dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                      int(bool(causal)), _default_scale(d, scale),
                                      workspace.data_ptr(),
                                      workspace.numel() * workspace.element_size(),
                                      _stream(stream))
    _check("attn_bwd_main", st)


def attn_bwd_main_dkdv(q, k, v, do, dk, dv, causal: bool, workspace, scale=None, stream=None):
    B, H, N, d = _shape4(q, "q")
    st = load_library().attn_bwd_main_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           do.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N,
                                           d, int(bool(causal)), _default_scale(d, scale),
                                           workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(stream))
    _check("attn_bwd_main_dkdv", st)


def attn_bwd_dq(q, k, v, do, dq, causal: bool, workspace, scale=None, stream=None):
    B, H, N, d = _shape4(q, "q")
    st = load_library().attn_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                    dq.data_ptr(), B, H, N, d, int(bool(causal)),
                                    _default_scale(d, scale), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check("attn_bwd_dq", st)


def attn_bwd_dq_convert(dq, workspace, scale=None, stream=None):
    B, H, N, d = _shape4(dq, "dq")
    st = load_library().attn_bwd_dq_convert(dq.data_ptr(), B, H, N, d, _default_scale(d, scale),
                                            workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(),
                                            _stream(stream))
    _check("attn_bwd_dq_convert", st)


def attn_last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load_library().attn_last_device_error(_stream(stream)))


def attn_device_error_word(stream=None):
    w = ctypes.c_int(0)
    st = load_library().attn_device_error_word(_stream(stream), ctypes.byref(w))
    return int(st), int(w.value)


def attn_watchdog_selftest(limit_ns: int, stream=None) -> int:
    return int(load_library().attn_watchdog_selftest(int(limit_ns), _stream(stream)))


# ------------------------------------------------------------------ Mamba-2 layer
def _ssd_dims(x, B):
    if x.dim() != 4 or B.dim() != 4:
        raise ValueError("x must be [Bt, T, H, P] and B [Bt, T, G, N]")
    Bt, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    return Bt, T, H, G, N, P


def ssd_workspace(Bt, T, H, G, N, P, device) -> torch.Tensor:
    n = max(int(load_library().ssd_workspace_size(Bt, T, H, G, N, P)), 256)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _ssd_check_inputs(x, dt, A, B, C, D, dims):
    Bt, T, H, G, N, P = dims
    _check_tensor(x, "x", (Bt, T, H, P))
    _check_tensor(B, "B", (Bt, T, G, N))
    _check_tensor(C, "C", (Bt, T, G, N))
    _check_tensor(dt, "dt", (Bt, T, H), torch.float32)
    _check_tensor(A, "A", (H,), torch.float32)
    _check_tensor(D, "D", (H,), torch.float32)


def ssd_fwd(x, dt, A, B, C, D, y=None, workspace=None, stream=None):
    """y [Bt, T, H, P] fp32 of the Mamba-2 state-space layer."""
    dims = _ssd_dims(x, B)
    _ssd_check_inputs(x, dt, A, B, C, D, dims)
    y = torch.empty(x.shape, dtype=torch.float32, device=x.device) if y is None else y
    _check_tensor(y, "y", x.shape, torch.float32)
    ws = ssd_workspace(*dims, x.device) if workspace is None else workspace
    st = load_library().ssd_fwd(x.data_ptr(), dt.data_ptr(), A.data_ptr(), B.data_ptr(),
                                C.data_ptr(), D.data_ptr(), y.data_ptr(), *dims, ws.data_ptr(),
                                ws.numel() * ws.element_size(), _stream(stream))
    _check("ssd_fwd", st)
    return y


def ssd_bwd(x, dt, A, B, C, D, dy, workspace=None, out=None, stream=None):
    """Gradients of <dy, y>: dict with dx, ddt, dA, dB, dC, dD (fp32)."""
    dims = _ssd_dims(x, B)
    _ssd_check_inputs(x, dt, A, B, C, D, dims)
    _check_tensor(dy, "dy", x.shape)
    f32 = dict(dtype=torch.float32, device=x.device)
    if out is None:
        out = {"dx": torch.empty(x.shape, **f32), "ddt": torch.empty(dt.shape, **f32),
               "dA": torch.empty(A.shape, **f32), "dB": torch.empty(B.shape, **f32),
               "dC": torch.empty(C.shape, **f32), "dD": torch.empty(D.shape, **f32)}
    ws = ssd_workspace(*dims, x.device) if workspace is None else workspace
    st = load_library().ssd_bwd(x.data_ptr(), dt.data_ptr(), A.data_ptr(), B.data_ptr(),
                                C.data_ptr(), D.data_ptr(), dy.data_ptr(), out["dx"].data_ptr(),
                                out["ddt"].data_ptr(), out["dA"].data_ptr(),
                                out["dB"].data_ptr(), out["dC"].data_ptr(),
                                out["dD"].data_ptr(), *dims, ws.data_ptr(),
                                ws.numel() * ws.element_size(), _stream(stream))
    _check("ssd_bwd", st)
    return out
