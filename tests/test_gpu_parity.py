"""CUDA path against the fp64 oracle on the same seeded bf16 inputs.

Tolerance: for each of O, dQ, dK, dV, max|gpu - oracle| / max|oracle| <= 1e-2
(bf16 inputs and outputs, fp32 accumulation).  L is checked as an absolute
error (it is a log, O(1)-sized): <= 2e-2.

* All five named workloads are compared element by element over the whole
  tensors, the three large ones (N = 4096 .. 16384, d = 128) at full size in
  the benchmark's launch configuration.
* Ragged lengths (N not a multiple of the 128-row tile, N < 128, N = 1),
  both head dims, both mask modes.
* Degenerate inputs: Q = 0 (uniform softmax), sharpened Q, empty problems.
* The backward fed with the oracle's own O and L (backward-only parity).
* Determinism, the three backward steps against the one-call backward, and
  the bounded-wait failure path.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import WORKLOADS, make_inputs, make_tensor

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


def assert_no_device_error(what=""):
    st, word = ab.attn_device_error_word()
    assert st == ab.ATTN_OK, "%s: device error status %d, word 0x%08x" % (what, st, word)


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


def gpu_fwd_bwd(q, k, v, do, causal, scale, dq_method=ab.ATTN_DQ_AUTO):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o, lse = ab.attn_fwd(qd, kd, vd, causal, scale)
    dq, dk, dv = ab.attn_bwd(qd, kd, vd, o, dod, lse, causal, scale, dq_method=dq_method)
    torch.cuda.synchronize()
    return dict(O=o, L=lse, dQ=dq, dK=dk, dV=dv)


def check_full(gpu, ref, what):
    errs = {name: rel_err(gpu[name], ref[name]) for name in ("O", "dQ", "dK", "dV")}
    lerr = float(np.max(np.abs(f64(gpu["L"]) - ref["L"]))) if ref["L"].size else 0.0
    msg = "%s: %s, L abs %.2e" % (what, {k: "%.2e" % v for k, v in errs.items()}, lerr)
    assert all(e <= TOL for e in errs.values()), msg
    assert lerr <= L_ATOL, msg
    return errs


@pytest.mark.parametrize("name", ["b1h2n128d64", "b2h16n2048d64_causal"])
def test_workload_full_tensors(name):
    """Both ways of forming dQ (reduce-add into an accumulator; the separate
    query-stationary pass) against the same oracle result."""
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    ref = oracle.attention_forward_backward(q, k, v, do, w.causal, w.scale)
    for mname, method in METHODS.items():
        gpu = gpu_fwd_bwd(q, k, v, do, w.causal, w.scale, method)
        check_full(gpu, ref, "%s dq=%s" % (name, mname))
        assert_no_device_error("%s dq=%s" % (name, mname))


@pytest.mark.parametrize("name", ["b1h2n128d64", "b2h16n2048d64_causal"])
def test_backward_only_from_oracle_forward(name):
    """The backward alone, fed with bf16(O_oracle) and fp32(L_oracle)."""
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    ref = oracle.attention_forward_backward(q, k, v, do, w.causal, w.scale)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.from_numpy(ref["O"]).to(torch.bfloat16).to(dev)
    lse = torch.from_numpy(ref["L"]).to(torch.float32).to(dev)
    dq, dk, dv = ab.attn_bwd(qd, kd, vd, o, dod, lse, w.causal, w.scale)
    torch.cuda.synchronize()
    for g, r, n in ((dq, ref["dQ"], "dQ"), (dk, ref["dK"], "dK"), (dv, ref["dV"], "dV")):
        e = rel_err(g, r)
        assert e <= TOL, "%s %s %.2e" % (name, n, e)


@pytest.mark.parametrize("name", ["b1h32n4096d128_causal", "b4h16n8192d128",
                                  "b1h16n16384d128_causal"])
def test_workload_full_size_full_tensors(name):
    """The three large named workloads at full size, in the benchmark's launch
    configuration, compared with the oracle element by element over the whole
    O, L, dQ, dK and dV tensors (every head, so every work-item group of the
    persistent backward and its boundaries).  The oracle takes about 10 s,
    140 s and 70 s for these on 16 host cores."""
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    runs = {}
    for mname, method in METHODS.items():
        runs[mname] = {n: t.cpu() for n, t in
                       gpu_fwd_bwd(q, k, v, do, w.causal, w.scale, method).items()}
        assert_no_device_error("%s dq=%s" % (name, mname))
        torch.cuda.empty_cache()
    ref = oracle.attention_forward_backward(q, k, v, do, w.causal, w.scale)
    for mname, gpu in runs.items():
        what = "%s dq=%s" % (name, mname)
        errs = check_full(gpu, ref, what)
        # per-head worst error, so a failure names the head
        for hname in ("dQ", "dK", "dV"):
            g = f64(gpu[hname]).reshape(w.heads, -1)
            r = ref[hname].reshape(w.heads, -1)
            worst = np.max(np.abs(g - r), axis=1) / np.max(np.abs(r))
            assert np.all(worst <= TOL), "%s %s: worst head %d (%.2e)" % (
                what, hname, int(np.argmax(worst)), float(np.max(worst)))
        assert max(errs.values()) <= TOL


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 100, 128, 129, 255, 256, 300, 384, 513])
def test_ragged_lengths(N, d, causal):
    B, H = 1, 3
    seed = 1000 + N * 4 + (d // 64) * 2 + int(causal)
    q, k, v, do = (make_tensor((B, H, N, d), seed + 7919 * i) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_forward_backward(q, k, v, do, causal, scale)
    for mname, method in METHODS.items():
        gpu = gpu_fwd_bwd(q, k, v, do, causal, scale, method)
        check_full(gpu, ref, "N=%d d=%d causal=%s dq=%s" % (N, d, causal, mname))


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("d", [64, 128])
def test_many_tasks_per_cta_ragged(d, causal):
    """More (head, query-tile pair) tasks than SMs but fewer than two per SM
    (the forward's grid is then persistent with or without the causal mask),
    half of them without a second query tile (N = 300: tiles of 128, 128 and
    44 rows), so that forward CTAs run tasks of both kinds in turn."""
    B, H, N = 2, 60, 300
    seed = 5100 + d + int(causal)
    q, k, v, do = (make_tensor((B, H, N, d), seed + 7919 * i) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_forward_backward(q, k, v, do, causal, scale)
    gpu = gpu_fwd_bwd(q, k, v, do, causal, scale)
    check_full(gpu, ref, "B=%d H=%d N=%d d=%d causal=%s" % (B, H, N, d, causal))


@pytest.mark.parametrize("d", [64, 128])
def test_zero_queries_uniform_softmax(d):
    """Q = 0: P is uniform over the visible keys; O is a (prefix) mean of V."""
    B, H, N = 2, 2, 320
    k, v, do = (make_tensor((B, H, N, d), 31 + i) for i in range(3))
    q = torch.zeros_like(k)
    for causal in (False, True):
        ref = oracle.attention_forward_backward(q, k, v, do, causal, 1 / math.sqrt(d))
        for mname, method in METHODS.items():
            gpu = gpu_fwd_bwd(q, k, v, do, causal, 1 / math.sqrt(d), method)
            check_full(gpu, ref, "Q=0 d=%d causal=%s dq=%s" % (d, causal, mname))


@pytest.mark.parametrize("qscale", [4.0, 8.0])
def test_sharp_softmax(qscale):
    """Large logits: the online maximum moves many times and P is peaky."""
    B, H, N, d = 1, 4, 640, 128
    q = make_tensor((B, H, N, d), 41, std=qscale)
    k, v, do = (make_tensor((B, H, N, d), 42 + i) for i in range(3))
    for causal in (False, True):
        ref = oracle.attention_forward_backward(q, k, v, do, causal, 1 / math.sqrt(d))
        for mname, method in METHODS.items():
            gpu = gpu_fwd_bwd(q, k, v, do, causal, 1 / math.sqrt(d), method)
            check_full(gpu, ref, "sharp %g causal=%s dq=%s" % (qscale, causal, mname))


def test_non_default_scale():
    B, H, N, d = 1, 2, 384, 64
    q, k, v, do = (make_tensor((B, H, N, d), 51 + i) for i in range(4))
    for scale in (0.02, 0.5):
        ref = oracle.attention_forward_backward(q, k, v, do, True, scale)
        for mname, method in METHODS.items():
            gpu = gpu_fwd_bwd(q, k, v, do, True, scale, method)
            check_full(gpu, ref, "scale %g dq=%s" % (scale, mname))


def test_empty_problem():
    dev = torch.device("cuda", 0)
    z = torch.empty((2, 3, 0, 64), dtype=torch.bfloat16, device=dev)
    o, lse = ab.attn_fwd(z, z, z, True)
    dq, dk, dv = ab.attn_bwd(z, z, z, o, z, lse, True)
    assert o.shape == (2, 3, 0, 64) and lse.shape == (2, 3, 0) and dq.numel() == 0


def test_steps_match_one_call_and_determinism():
    w = WORKLOADS["b2h16n2048d64_causal"]
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    o1, l1 = ab.attn_fwd(q, k, v, True)
    o2, l2 = ab.attn_fwd(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2), "forward is deterministic"
    dq1, dk1, dv1 = ab.attn_bwd(q, k, v, o1, do, l1, True)
    ws = ab.alloc_workspace(w.B, w.H, w.N, w.d, dev)
    dq2, dk2, dv2 = (torch.empty_like(q) for _ in range(3))
    ab.attn_bwd_preprocess(o1, do, l1, ws)
    ab.attn_bwd_main(q, k, v, do, dk2, dv2, True, ws)
    ab.attn_bwd_dq_convert(dq2, ws)
    torch.cuda.synchronize()
    # dK and dV are accumulated in tensor memory by one CTA: bitwise repeatable.
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    # dQ is summed with fp32 atomics across CTAs: equal up to summation order.
    assert rel_err(dq2, f64(dq1)) <= 2e-3


def test_separate_dq_steps_and_determinism():
    """The separate-pass backward equals its three steps run one by one, and
    every output, dQ included, is bitwise repeatable (no cross-CTA sums)."""
    w = WORKLOADS["b2h16n2048d64_causal"]
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    o, lse = ab.attn_fwd(q, k, v, True)
    sep = ab.ATTN_DQ_SEPARATE
    dq1, dk1, dv1 = ab.attn_bwd(q, k, v, o, do, lse, True, dq_method=sep)
    dq2, dk2, dv2 = ab.attn_bwd(q, k, v, o, do, lse, True, dq_method=sep)
    ws = ab.alloc_workspace(w.B, w.H, w.N, w.d, dev)
    dq3, dk3, dv3 = (torch.empty_like(q) for _ in range(3))
    ab.attn_bwd_preprocess(o, do, lse, ws)
    ab.attn_bwd_main_dkdv(q, k, v, do, dk3, dv3, True, ws)
    ab.attn_bwd_dq(q, k, v, do, dq3, True, ws)
    dq4, dk4, dv4 = ab.attn_bwd(q, k, v, o, do, lse, True, dq_method=ab.ATTN_DQ_REDUCE)
    torch.cuda.synchronize()
    for a, b_, c in ((dq1, dq2, dq3), (dk1, dk2, dk3), (dv1, dv2, dv3)):
        assert torch.equal(a, b_) and torch.equal(a, c)
    # dK, dV come from the same arithmetic in both main-kernel families
    assert torch.equal(dk1, dk4) and torch.equal(dv1, dv4)
    # dQ: one bf16 rounding of a different fp32 summation order
    assert rel_err(dq1, f64(dq4)) <= 2e-3


def test_watchdog_reports_timeout_without_fault():
    """A wait nothing can satisfy gives up after its limit and reports
    ATTN_ERR_TIMEOUT; the context stays usable."""
    assert ab.attn_last_device_error() == ab.ATTN_OK
    assert ab.attn_watchdog_selftest(20_000_000) == ab.ATTN_OK
    st, word = ab.attn_device_error_word()
    assert st == ab.ATTN_ERR_TIMEOUT and (word >> 24) == 1 and (word & 0xFFFFFF) == 0xD06
    assert ab.attn_last_device_error() == ab.ATTN_OK  # cleared
    w = WORKLOADS["b1h2n128d64"]
    q, k, v, do = make_inputs(w)
    ref = oracle.attention_forward_backward(q, k, v, do, w.causal, w.scale)
    check_full(gpu_fwd_bwd(q, k, v, do, w.causal, w.scale), ref, "after watchdog")
