"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
function include/attn.h declares, and validates arguments on the host
(documented statuses, nothing launched).  CPU only."""

import ctypes
import os
import re

import pytest

from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300 import build as abuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    abuild.build()
    return ab.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size",
                     "attn_last_device_error", "attn_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), "missing export %s" % name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_no_undeclared_attn_exports(lib):
    # every binding signature corresponds to a declaration
    names = set(declared_functions())
    for name in ("attn_fwd", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_main",
                 "attn_bwd_dq_convert", "attn_device_error_word", "attn_watchdog_selftest",
                 "attn_version"):
        assert name in names


def test_status_strings(lib):
    for st in range(7):
        assert lib.attn_status_string(st)
    assert lib.attn_status_string(99) == b"unknown status"
    assert lib.attn_version() >= 100


def test_workspace_size(lib):
    # D and L2: BH*Npad fp32 each; acc: BH*Npad*d fp32; two int32 per tile and
    # one per row for document ranges; each section 256-aligned
    def expect(B, H, N, d):
        npad = (N + 127) // 128 * 128
        r = lambda x: (x + 255) // 256 * 256
        return (3 * r(4 * B * H * npad) + r(4 * B * H * npad * d)
                + r(8 * B * H * (npad // 128)) + r(4 * B * H * (npad // 128)))
    for args in ((1, 2, 128, 64), (2, 16, 2048, 64), (1, 3, 129, 128), (4, 16, 8192, 128)):
        assert lib.attn_bwd_workspace_size(*args) == expect(*args)
    assert lib.attn_bwd_workspace_size(0, 2, 128, 64) == 0
    assert lib.attn_bwd_workspace_size(1, 2, 0, 64) == 0
    assert lib.attn_bwd_workspace_size(1, 2, 128, 96) == 0
    assert lib.attn_bwd_workspace_size(-1, 2, 128, 64) == 0


FAKE = 0x10000  # a 16-byte aligned non-null address; never dereferenced


def fwd(lib, Q=FAKE, K=FAKE, V=FAKE, O=FAKE, L=FAKE, B=1, H=1, N=128, d=64, causal=0, scale=0.125):
    return lib.attn_fwd(Q, K, V, O, L, B, H, N, d, causal, scale, None)


def bwd(lib, ptr=FAKE, B=1, H=1, N=128, d=64, causal=0, scale=0.125, ws=FAKE, wsb=None):
    if wsb is None:
        wsb = lib.attn_bwd_workspace_size(max(B, 0), max(H, 0), max(N, 0), d)
    return lib.attn_bwd(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, B, H, N, d, causal, scale,
                        ws, wsb, None)


def test_fwd_validation(lib):
    assert fwd(lib, Q=None) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, L=None) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, V=FAKE + 8) == ab.ATTN_ERR_INVALID_ARG       # misaligned
    assert fwd(lib, B=-1) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, N=-5) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, d=96) == ab.ATTN_ERR_UNSUPPORTED
    assert fwd(lib, d=256) == ab.ATTN_ERR_UNSUPPORTED
    assert fwd(lib, causal=2) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, scale=0.0) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, scale=-1.0) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, scale=float("nan")) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, scale=float("inf")) == ab.ATTN_ERR_INVALID_ARG
    assert fwd(lib, B=1 << 20, H=1 << 12) == ab.ATTN_ERR_UNSUPPORTED  # rows beyond 31 bits
    # empty problems are valid and launch nothing, even with null pointers
    assert fwd(lib, Q=None, K=None, V=None, O=None, L=None, N=0) == ab.ATTN_OK
    assert fwd(lib, Q=None, K=None, V=None, O=None, L=None, B=0) == ab.ATTN_OK


def test_bwd_validation(lib):
    assert bwd(lib, ptr=None) == ab.ATTN_ERR_INVALID_ARG
    assert bwd(lib, d=32) == ab.ATTN_ERR_UNSUPPORTED
    assert bwd(lib, H=-2) == ab.ATTN_ERR_INVALID_ARG
    assert bwd(lib, scale=0.0) == ab.ATTN_ERR_INVALID_ARG
    assert bwd(lib, ws=None) == ab.ATTN_ERR_WORKSPACE
    assert bwd(lib, ws=FAKE + 16) == ab.ATTN_ERR_WORKSPACE               # not 256-aligned
    need = lib.attn_bwd_workspace_size(1, 1, 128, 64)
    assert bwd(lib, wsb=need - 1) == ab.ATTN_ERR_WORKSPACE
    assert bwd(lib, ptr=None, ws=None, wsb=0, N=0) == ab.ATTN_OK
    # the three steps validate the same way
    assert lib.attn_bwd_preprocess(FAKE, FAKE, None, 1, 1, 128, 64, FAKE, need, None) == \
        ab.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_preprocess(FAKE, FAKE, FAKE, 1, 1, 128, 64, FAKE, 0, None) == \
        ab.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_main(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 128, 1, -0.5,
                             FAKE, need, None) == ab.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_dq_convert(None, 1, 1, 128, 64, 0.125, FAKE, need, None) == \
        ab.ATTN_ERR_INVALID_ARG
    assert lib.attn_watchdog_selftest(10, None) == ab.ATTN_ERR_INVALID_ARG


def test_dq_method_and_split_steps_validation(lib):
    """attn_bwd_opts takes only the three documented dQ methods; the two steps
    of the separate-pass backward validate like the other steps."""
    need = lib.attn_bwd_workspace_size(1, 1, 128, 64)

    def opts(method, N=128, ptr=FAKE):
        return lib.attn_bwd_opts(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, N, 64, 1, 0,
                                 None, 0.125, method, FAKE, need, None)
    for bad in (-1, 3, 99):
        assert opts(bad) == ab.ATTN_ERR_INVALID_ARG
        assert opts(bad, N=0, ptr=None) == ab.ATTN_ERR_INVALID_ARG
    for good in (ab.ATTN_DQ_AUTO, ab.ATTN_DQ_REDUCE, ab.ATTN_DQ_SEPARATE):
        assert opts(good, N=0, ptr=None) == ab.ATTN_OK
        assert opts(good, ptr=None) == ab.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_main_dkdv(FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 1, 128, 64, 1, 0.125,
                                  FAKE, need, None) == ab.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_main_dkdv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 96, 1, 0.125,
                                  FAKE, need, None) == ab.ATTN_ERR_UNSUPPORTED
    assert lib.attn_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128, 64, 1, 0.125, FAKE, need - 1,
                           None) == ab.ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE + 8, 1, 1, 128, 64, 1, 0.125, FAKE, need,
                           None) == ab.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_dq(None, None, None, None, None, 1, 1, 0, 64, 1, 0.125, None, 0,
                           None) == ab.ATTN_OK


def test_fp8_forward_validation(lib):
    """attn_fwd_fp8: head dim 128 only; every descale factor finite and > 0;
    pointers checked like attn_fwd's; an empty problem launches nothing."""
    def f8(ptr=FAKE, N=128, d=128, causal=0, qd=1.0, kd=1.0, vd=1.0, scale=0.125, q=None):
        return lib.attn_fwd_fp8(ptr if q is None else q, ptr, ptr, qd, kd, vd, ptr, ptr, 1, 2, N,
                                d, causal, scale, None)
    assert f8(d=64) == ab.ATTN_ERR_UNSUPPORTED
    assert f8(d=96) == ab.ATTN_ERR_UNSUPPORTED
    assert f8(qd=0.0) == ab.ATTN_ERR_INVALID_ARG
    assert f8(kd=float("inf")) == ab.ATTN_ERR_INVALID_ARG
    assert f8(vd=float("nan")) == ab.ATTN_ERR_INVALID_ARG
    assert f8(qd=1e30, kd=1e30) == ab.ATTN_ERR_INVALID_ARG  # combined score scale overflows
    assert f8(scale=-1.0) == ab.ATTN_ERR_INVALID_ARG
    assert f8(causal=5) == ab.ATTN_ERR_INVALID_ARG
    assert f8(q=0) == ab.ATTN_ERR_INVALID_ARG
    assert f8(q=FAKE + 4) == ab.ATTN_ERR_INVALID_ARG
    assert f8(ptr=None, N=0) == ab.ATTN_OK


def test_ssd_validation(lib):
    """The Mamba-2 layer: P = 64 and N in {64, 128} only, heads a multiple of
    groups, pointers and workspace checked before any launch."""
    ws_need = lib.ssd_workspace_size(1, 128, 2, 1, 128, 64)
    assert ws_need > 0 and ws_need % 4 == 0
    assert lib.ssd_workspace_size(1, 128, 2, 1, 128, 32) == 0
    assert lib.ssd_workspace_size(1, 0, 2, 1, 128, 64) == 0

    def bwd_(Bt=1, T=128, H=2, G=1, N=128, P=64, ptr=FAKE, ws=FAKE, wsb=None, dt=FAKE):
        wsb = ws_need if wsb is None else wsb
        return lib.ssd_bwd(ptr, dt, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr,
                           Bt, T, H, G, N, P, ws, wsb, None)
    assert bwd_(P=32) == ab.ATTN_ERR_UNSUPPORTED
    assert bwd_(N=96) == ab.ATTN_ERR_UNSUPPORTED
    assert bwd_(H=3, G=2) == ab.ATTN_ERR_INVALID_ARG
    assert bwd_(G=0) == ab.ATTN_ERR_INVALID_ARG
    assert bwd_(T=-1) == ab.ATTN_ERR_INVALID_ARG
    assert bwd_(ptr=None) == ab.ATTN_ERR_INVALID_ARG
    assert bwd_(dt=FAKE + 2) == ab.ATTN_ERR_INVALID_ARG
    assert bwd_(ws=None) == ab.ATTN_ERR_WORKSPACE
    assert bwd_(wsb=ws_need - 4) == ab.ATTN_ERR_WORKSPACE
    assert bwd_(ptr=None, T=0, ws=None, wsb=0, dt=None) == ab.ATTN_OK
    assert lib.ssd_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 128, 2, 1, 128, 64, FAKE,
                       ws_need, None) == ab.ATTN_ERR_INVALID_ARG


def test_fp8_backward_validation(lib):
    """attn_bwd_fp8: head dim 128 only, every factor finite and > 0, pointers,
    workspace and the amax word checked before any launch."""
    need = lib.attn_bwd_workspace_size(1, 2, 128, 128)

    def b8(d=128, N=128, ptr=FAKE, ds=1.0, qd=1.0, amax=None, ws=FAKE, wsb=None, causal=1):
        return lib.attn_bwd_fp8(ptr, ptr, ptr, ptr, ptr, ptr, qd, 1.0, 1.0, 1.0, ds, ptr, ptr, ptr,
                                amax, 1, 2, N, d, causal, 0.088, ws, need if wsb is None else wsb,
                                None)
    assert b8(d=64) == ab.ATTN_ERR_UNSUPPORTED
    assert b8(ds=0.0) == ab.ATTN_ERR_INVALID_ARG
    assert b8(ds=float("nan")) == ab.ATTN_ERR_INVALID_ARG
    assert b8(qd=-1.0) == ab.ATTN_ERR_INVALID_ARG
    assert b8(amax=FAKE + 2) == ab.ATTN_ERR_INVALID_ARG
    assert b8(ptr=None) == ab.ATTN_ERR_INVALID_ARG
    assert b8(ws=None) == ab.ATTN_ERR_WORKSPACE
    assert b8(wsb=need - 1) == ab.ATTN_ERR_WORKSPACE
    assert b8(causal=2) == ab.ATTN_ERR_INVALID_ARG
    assert b8(ptr=None, N=0, ws=None, wsb=0) == ab.ATTN_OK


def test_noalloc_passes_argument_errors_through(lib):
    """attn_bwd_noalloc answers every bad argument the way attn_bwd does, before
    it looks up its scratch (nothing here reaches the GPU): an unsupported head
    dim, a null or misaligned pointer, a bad scale, and an empty problem, which
    is valid and launches nothing."""
    def noalloc(ptr=FAKE, B=1, H=1, N=128, d=64, causal=0, scale=0.125, q=None):
        qp = ptr if q is None else q
        return lib.attn_bwd_noalloc(qp, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, B, H, N, d,
                                    causal, scale, None)
    assert noalloc(d=96) == ab.ATTN_ERR_UNSUPPORTED
    assert noalloc(ptr=None) == ab.ATTN_ERR_INVALID_ARG
    assert noalloc(q=FAKE + 8) == ab.ATTN_ERR_INVALID_ARG   # misaligned Q
    assert noalloc(q=0) == ab.ATTN_ERR_INVALID_ARG          # null Q only
    assert noalloc(scale=0.0) == ab.ATTN_ERR_INVALID_ARG
    assert noalloc(causal=3) == ab.ATTN_ERR_INVALID_ARG
    assert noalloc(B=-1) == ab.ATTN_ERR_INVALID_ARG
    assert noalloc(ptr=None, B=0) == ab.ATTN_OK
    assert noalloc(ptr=None, N=0) == ab.ATTN_OK


def test_window_validation(lib):
    """The sliding window is causal only and non-negative; checked before
    anything else is looked at, empty problems included."""
    def fwd_ex(causal, window, N=128, ptr=FAKE, doc=None):
        return lib.attn_fwd_ex(ptr, ptr, ptr, ptr, ptr, 1, 1, N, 64, causal, window, doc, 0.125,
                               None)

    def bwd_ex(causal, window, N=128, ptr=FAKE, doc=None):
        need = lib.attn_bwd_workspace_size(1, 1, max(N, 0), 64)
        return lib.attn_bwd_ex(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 1, N, 64, causal,
                               window, doc, 0.125, FAKE, need, None)
    for f in (fwd_ex, bwd_ex):
        assert f(0, 16) == ab.ATTN_ERR_INVALID_ARG
        assert f(1, -1) == ab.ATTN_ERR_INVALID_ARG
        assert f(0, 16, N=0, ptr=None) == ab.ATTN_ERR_INVALID_ARG
        assert f(1, 16, N=0, ptr=None) == ab.ATTN_OK
        assert f(1, 16, ptr=None) == ab.ATTN_ERR_INVALID_ARG  # null pointers still rejected
        # document maps: causal only, 4-byte aligned
        assert f(0, 0, doc=FAKE) == ab.ATTN_ERR_INVALID_ARG
        assert f(1, 0, doc=FAKE + 2) == ab.ATTN_ERR_INVALID_ARG
        assert f(1, 0, N=0, ptr=None, doc=FAKE) == ab.ATTN_OK


def test_binding_checks_tensors():
    import torch

    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ab.attn_fwd(q, q, q, causal=False)  # CPU tensors are rejected, nothing falls back


def test_missing_library_raises(tmp_path):
    """Without the built CUDA library the binding raises; there is no other path."""
    with pytest.raises(RuntimeError, match="not built"):
        ab.load_library(str(tmp_path / "libattn_gb300.so"))
