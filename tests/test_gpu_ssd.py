"""The Mamba-2 state-space layer (forward and backward) on the GPU against
the fp64 oracle (``oracle/ssd_oracle.c``: the recurrence and its adjoint).

Inputs are the same bf16/fp32 values on both sides.  The GPU computes in
fp32 (chunks of 64 steps, a scan over chunks), the oracle in fp64 step by
step, so the outputs differ by fp32 rounding only: sums of up to T*N terms
with unit roundoff 2^-24 (a random-walk growth of about sqrt(T N) 2^-24,
1e-4 at T N = 2^20 with a margin for cancellation) and the exponentials'
argument rounding (|dt A| summed over a chunk, times 2^-24).  Each output
array must satisfy max|gpu - oracle| <= 1e-4 * max|oracle| (dA and dD: per
head, against the largest |value| over the heads).  Measured: 1e-6 or less
at T = 2048.
"""

import numpy as np
import pytest
import torch

from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import (SSD_WORKLOADS, SsdWorkload,
                                                       make_ssd_inputs)
from oracle import ssd

pytestmark = pytest.mark.gpu

TOL = 1e-4
NAMES = ("dx", "ddt", "dA", "dB", "dC", "dD")


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


def rel(g, r):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert g.shape == r.shape and np.all(np.isfinite(g))
    den = float(np.max(np.abs(r))) if r.size else 0.0
    return float(np.max(np.abs(g - r)) / den) if den > 0 else float(np.max(np.abs(g), initial=0))


def run_gpu(inputs, backward=True):
    dev = torch.device("cuda", 0)
    x, dt, A, B, C, D, dy = (t.to(dev) for t in inputs)
    y = ab.ssd_fwd(x, dt, A, B, C, D)
    out = ab.ssd_bwd(x, dt, A, B, C, D, dy) if backward else {}
    torch.cuda.synchronize()
    st, word = ab.attn_device_error_word()
    assert st == ab.ATTN_OK, "device error %d word 0x%08x" % (st, word)
    res = {k: v.cpu().numpy().astype(np.float64) for k, v in out.items()}
    res["y"] = y.cpu().numpy().astype(np.float64)
    return res


def check(w, what):
    inputs = make_ssd_inputs(w)
    gpu = run_gpu(inputs)
    ref = ssd.ssd_forward_backward(*inputs)
    errs = {"y": rel(gpu["y"], ref["y"])}
    errs.update({n: rel(gpu[n], ref[n]) for n in NAMES})
    msg = "%s: %s" % (what, {k: "%.2e" % v for k, v in errs.items()})
    assert all(e <= TOL for e in errs.values()), msg
    return errs


@pytest.mark.parametrize("Bt,T,H,G,N", [(1, 64, 2, 1, 64), (2, 200, 4, 2, 64), (1, 1, 2, 1, 128),
                                        (1, 130, 2, 2, 128), (2, 1000, 4, 1, 128),
                                        (1, 63, 3, 3, 64), (1, 129, 2, 1, 128)])
def test_ssd_small_full_tensors(Bt, T, H, G, N):
    """Single and ragged chunks, several chunks, groups of one to three heads,
    both state sizes."""
    w = SsdWorkload("t", Bt, T, H, G, N, 64, seed=500 + T + 7 * H + N)
    check(w, "Bt=%d T=%d H=%d G=%d N=%d" % (Bt, T, H, G, N))


@pytest.mark.parametrize("name", sorted(SSD_WORKLOADS))
def test_ssd_workloads_full_tensors(name):
    """The named layer shapes (d_model 2048, 64 heads, state 128) at full size,
    every output element against the oracle."""
    check(SSD_WORKLOADS[name], name)


def test_ssd_repeatable_and_no_stale_state():
    """Every output is bitwise repeatable (each element has one writer, and
    the sums over heads, batches and chunks run in a fixed order), with the
    same workspace and output buffers reused after a call on different
    inputs (the gradients are overwritten, not accumulated into)."""
    dev = torch.device("cuda", 0)
    ws = ab.ssd_workspace(2, 300, 4, 2, 128, 64, dev)
    out = None
    res = []
    for seed in (77, 78, 77):
        x, dt, A, B, C, D, dy = (t.to(dev) for t in make_ssd_inputs(
            SsdWorkload("r", 2, 300, 4, 2, 128, 64, seed=seed)))
        out = ab.ssd_bwd(x, dt, A, B, C, D, dy, workspace=ws, out=out)
        torch.cuda.synchronize()
        res.append({k: v.cpu().numpy().astype(np.float64) for k, v in out.items()})
    a, b = res[0], res[2]
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        assert np.array_equal(a[k], b[k]), k
    assert ab.attn_last_device_error() == ab.ATTN_OK
