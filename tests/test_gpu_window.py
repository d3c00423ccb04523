"""Sliding-window (banded causal) attention on the GPU against the fp64
oracle: key j is visible to query i when i - window < j <= i.

Full tensors on ragged lengths and windows that start, end and straddle
128-row tiles; sampled rows at a long-sequence size with a 4096-key window
(the Mistral 7B setting named by "Training - CUDA Moat Still Alive",
section on attention variants); the plain causal path for window >= N; and
argument checks.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import make_tensor

pytestmark = pytest.mark.gpu

TOL = 1e-2
L_ATOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_backward_pass_attn_gb300 import build as abuild

    abuild.build()
    ab.load_library()
    assert ab.attn_last_device_error() == ab.ATTN_OK
    yield
    assert ab.attn_last_device_error() == ab.ATTN_OK


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape
    assert np.all(np.isfinite(g)), "non-finite GPU values"
    denom = np.max(np.abs(ref)) if ref.size else 0.0
    return float(np.max(np.abs(g - ref)) / denom) if denom > 0 else float(np.max(np.abs(g)))


METHODS = {"reduce": ab.ATTN_DQ_REDUCE, "separate": ab.ATTN_DQ_SEPARATE}


def gpu_fwd_bwd(q, k, v, do, scale, window, dq_method=ab.ATTN_DQ_AUTO):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ab.attn_fwd(qd, kd, vd, True, scale, window=window)
    dq, dk, dv = ab.attn_bwd(qd, kd, vd, o, dod, lse, True, scale, window=window,
                             dq_method=dq_method)
    torch.cuda.synchronize()
    return dict(O=o, L=lse, dQ=dq, dK=dk, dV=dv)


@pytest.mark.parametrize("method", sorted(METHODS))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,window", [(1, 1), (100, 1), (129, 64), (300, 128), (300, 129),
                                      (513, 200), (640, 256), (700, 511), (384, 383)])
def test_window_full_tensors(N, window, d, method):
    B, H = 1, 3
    seed = 5000 + N * 8 + window + d
    q, k, v, do = (make_tensor((B, H, N, d), seed + 7919 * i) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_forward_backward(q, k, v, do, True, scale, window=window)
    gpu = gpu_fwd_bwd(q, k, v, do, scale, window, METHODS[method])
    errs = {n: rel_err(gpu[n], ref[n]) for n in ("O", "dQ", "dK", "dV")}
    lerr = float(np.max(np.abs(f64(gpu["L"]) - ref["L"])))
    msg = "N=%d W=%d d=%d dq=%s: %s L %.2e" % (N, window, d, method, errs, lerr)
    assert all(e <= TOL for e in errs.values()), msg
    assert lerr <= L_ATOL, msg


def test_window_at_least_n_is_causal():
    """A window of N keys or more is the causal mask: the same bits."""
    B, H, N, d = 1, 2, 300, 64
    q, k, v, do = (make_tensor((B, H, N, d), 77 + i) for i in range(4))
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o1, l1 = ab.attn_fwd(qd, kd, vd, True)
    o2, l2 = ab.attn_fwd(qd, kd, vd, True, window=N)
    o3, l3 = ab.attn_fwd(qd, kd, vd, True, window=10 * N)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
    assert torch.equal(l1, l2) and torch.equal(l1, l3)
    g1 = ab.attn_bwd(qd, kd, vd, o1, dod, l1, True)
    g2 = ab.attn_bwd(qd, kd, vd, o1, dod, l1, True, window=N)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])  # dK, dV
    assert rel_err(g2[0], f64(g1[0])) <= 2e-3  # dQ: fp32 reductions, order may differ


@pytest.mark.parametrize("method", sorted(METHODS))
def test_window_long_sequence_sampled(method):
    """N = 16384, d = 128, a 4096-key window: sampled rows of two heads."""
    B, H, N, d, W = 1, 4, 16384, 128, 4096
    q, k, v, do = (make_tensor((B, H, N, d), 900 + i) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    gpu = gpu_fwd_bwd(q, k, v, do, scale, W, METHODS[method])
    rng = np.random.default_rng(5)
    for h in (0, H - 1):
        rows = sorted(set([0, 1, 127, 128, W - 1, W, W + 1, N // 2, N - 2, N - 1]
                          + rng.choice(N, 30, replace=False).tolist()))
        ref = oracle.attention_head_rows(q[0, h], k[0, h], v[0, h], do[0, h], True, scale,
                                         rows, rows, window=W)
        errs = {"O": rel_err(gpu["O"][0, h][rows], ref["O"]),
                "dQ": rel_err(gpu["dQ"][0, h][rows], ref["dQ"]),
                "dK": rel_err(gpu["dK"][0, h][rows], ref["dK"]),
                "dV": rel_err(gpu["dV"][0, h][rows], ref["dV"])}
        lerr = float(np.max(np.abs(f64(gpu["L"][0, h][rows]) - ref["L"])))
        msg = "head %d: %s L %.2e" % (h, errs, lerr)
        assert all(e <= TOL for e in errs.values()), msg
        assert lerr <= L_ATOL, msg


def test_window_argument_checks():
    dev = torch.device("cuda", 0)
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ab.AttnError) as e:
        ab.attn_fwd(q, q, q, False, window=16)  # the band is causal
    assert e.value.status == ab.ATTN_ERR_INVALID_ARG
    with pytest.raises(ab.AttnError) as e:
        ab.attn_fwd(q, q, q, True, window=-1)
    assert e.value.status == ab.ATTN_ERR_INVALID_ARG
