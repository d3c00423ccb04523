"""The e4m3 (fp8) backward on the GPU against the fp64 oracle.

The fp8 backward takes E4M3 Q, K, V, dO with one descale factor each; the
oracle decodes them (``oracle.fp8``) and runs its exact forward and backward
on those values.  The GPU backward is fed the oracle's own O (rounded to
bf16) and L, so what remains is the backward's own rounding:

* P is rounded to e4m3 as 256 P for dV; dS = P o (dP - D) is rounded to e4m3
  as ds_scale x dS for dK and dQ (P held in bf16 on the way: relative error
  below 2^-4 + 2^-9 per value), with absolute errors 2^-18 (P) and
  2^-10 / ds_scale (dS) below e4m3's normal range.  Treating the roundings as
  independent and uniform, element (j, c) of dV, dK and (i, c) of dQ has the
  variance
      dV: u^2/3 sum_i P_ij^2 dO_ic^2          + (2^-18)^2/3 n_j max dO_c^2
      dK: u^2/3 s^2 sum_i dS_ij^2 q_ic^2      + (2^-10/ds)^2/3 s^2 n_j max q_c^2
      dQ: u^2/3 s^2 sum_j dS_ij^2 k_jc^2      + (2^-10/ds)^2/3 s^2 N max k_c^2
  (u = 2^-4 + 2^-9; the sums from ``oracle.backward_rounding_budget``).
* D is formed from the bf16 O: |dD_i| <= 2^-9 sum_c |dO_ic O_ic|, a
  deterministic error that moves dK by at most s sum_i P_ij |dD_i| |q_ic| and
  dQ by at most s |dD_i| sum_j P_ij |k_jc| (the oracle's own backward and
  forward on those weights supply both sums).

Every element must satisfy |gpu - oracle| <= 7 sigma + (the D term) + 2^-8
|oracle| (bf16 outputs) + 1e-5 max|oracle|, and the root-mean-square error of
each output must stay within 1.5x the predicted one.  The dS scale is taken
the way fp8 training takes it: a first call reports max |dS|, and the call
under test uses the largest power of two with ds_scale x max|dS| <= 448.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import WORKLOADS, make_inputs, make_tensor, \
    quantize_e4m3

pytestmark = pytest.mark.gpu

U = 2.0 ** -4 + 2.0 ** -9


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


def run_case(q, k, v, do, causal, what):
    B, H, N, d = q.shape
    s = 1.0 / math.sqrt(d)
    (q8, qd), (k8, kd), (v8, vd), (do8, dod) = (quantize_e4m3(t) for t in (q, k, v, do))
    qf, kf, vf, dof = (fp8.dequantize(t8, sc) for t8, sc in
                       ((q8, qd), (k8, kd), (v8, vd), (do8, dod)))
    ref = oracle.attention_forward_backward(qf, kf, vf, dof, causal, s)
    dev = torch.device("cuda", 0)
    o_bf = torch.from_numpy(ref["O"]).to(torch.bfloat16)
    lse = torch.from_numpy(ref["L"]).to(torch.float32).to(dev)
    args = [t.to(dev) for t in (q8, k8, v8)] + [o_bf.to(dev), do8.to(dev), lse]
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    ab.attn_bwd_fp8(args[0], args[1], args[2], args[3], args[4], args[5], (qd, kd, vd, dod),
                    1.0, causal, s, ds_amax=amax)
    torch.cuda.synchronize()
    m = float(amax.item())
    assert m >= 0 and math.isfinite(m), "ds_amax %r" % m
    ds_scale = 2.0 ** math.floor(math.log2(448.0 / m)) if m > 0 else 1.0
    dq, dk, dv = ab.attn_bwd_fp8(args[0], args[1], args[2], args[3], args[4], args[5],
                                 (qd, kd, vd, dod), ds_scale, causal, s, ds_amax=amax)
    torch.cuda.synchronize()
    st, word = ab.attn_device_error_word()
    assert st == ab.ATTN_OK, "device error %d word 0x%08x" % (st, word)
    # the D term: dD_i <= 2^-9 sum_c |dO_ic O_ic|
    o_used = o_bf.to(torch.float64).numpy()
    dD = 2.0 ** -9 * np.sum(np.abs(dof * o_used), axis=-1)                # [B,H,N]
    # the reported maximum agrees with the oracle's max |dS| up to P's bf16
    # rounding (2^-8 relative, with a margin) and the D term (|P| <= 1)
    budget = oracle.backward_rounding_budget(qf, kf, vf, dof, causal, s, ref["L"], ref["D"])
    dsmax = float(np.max(budget["dsmax"]))
    assert abs(float(amax.item()) - dsmax) <= 0.02 * dsmax + float(np.max(dD)), \
        (amax.item(), dsmax)
    wK = oracle.attention_forward_backward(qf, kf, vf, dD[..., None] * np.abs(qf), causal,
                                           s)["dV"] * s   # sum_i P_ij |dD_i| |q_ic|
    wQ = s * dD[..., None] * oracle.attention_forward(qf, kf, np.abs(kf), causal, s)[0]
    n = budget["nvis"][..., None]
    out = {}
    for name, g, r, var, w in (
            ("dV", dv, ref["dV"], U * U / 3 * budget["vP"] +
             (2.0 ** -18) ** 2 / 3 * n * np.max(dof ** 2, axis=2, keepdims=True), 0.0),
            ("dK", dk, ref["dK"], U * U / 3 * s * s * budget["vK"] +
             (2.0 ** -10 / ds_scale) ** 2 / 3 * s * s * n * np.max(qf ** 2, axis=2, keepdims=True),
             wK),
            ("dQ", dq, ref["dQ"], U * U / 3 * s * s * budget["vQ"] +
             (2.0 ** -10 / ds_scale) ** 2 / 3 * s * s * N * np.max(kf ** 2, axis=2, keepdims=True),
             wQ)):
        gv = g.cpu().to(torch.float64).numpy()
        assert np.all(np.isfinite(gv)), "%s %s not finite" % (what, name)
        err = np.abs(gv - r)
        rmax = float(np.max(np.abs(r)))
        bound = 7 * np.sqrt(var) + w + 2.0 ** -8 * np.abs(r) + 1e-5 * rmax
        worst = float(np.max(err / bound))
        rms = float(np.sqrt(np.mean(err ** 2)))
        rms_pred = float(np.sqrt(np.mean(var + (2.0 ** -9 * r) ** 2 + np.square(w))))
        rel = float(np.max(err) / rmax) if rmax > 0 else float(np.max(err))
        msg = "%s %s: worst err/bound %.3f, rms %.3e (predicted %.3e), max|err|/max %.3e" % (
            what, name, worst, rms, rms_pred, rel)
        assert worst <= 1.0, msg
        assert rms <= 1.5 * rms_pred + 1e-9, msg
        out[name] = rel
    return out


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("N", [1, 100, 128, 300, 513])
def test_fp8_backward_ragged(N, causal):
    B, H, d = 1, 3, 128
    seed = 4000 + 2 * N + int(causal)
    q, k, v, do = (make_tensor((B, H, N, d), seed + 7919 * i) for i in range(4))
    run_case(q, k, v, do, causal, "N=%d causal=%s" % (N, causal))


def test_fp8_backward_sharp_softmax():
    B, H, N, d = 1, 2, 640, 128
    q = make_tensor((B, H, N, d), 71, std=4.0)
    k, v, do = (make_tensor((B, H, N, d), 72 + i) for i in range(3))
    for causal in (False, True):
        run_case(q, k, v, do, causal, "sharp causal=%s" % causal)


@pytest.mark.parametrize("name,batch,heads", [("b1h32n4096d128_causal", 1, 32),
                                              ("b4h16n8192d128", 1, 16),
                                              ("b1h16n16384d128_causal", 1, 4)])
def test_fp8_backward_workloads(name, batch, heads):
    """The d = 128 workloads quantised to e4m3, over whole tensors: the first
    at full size; the N = 8192 one with one batch element (its 16 heads) and
    the N = 16384 one with its first 4 heads, which keeps the oracle's share
    of the test within a few minutes."""
    w = WORKLOADS[name]
    q, k, v, do = (t[:batch, :heads].contiguous() for t in make_inputs(w))
    run_case(q, k, v, do, w.causal, "%s[:%d,:%d]" % (name, batch, heads))


def test_fp8_backward_argument_checks():
    dev = torch.device("cuda", 0)
    z = torch.zeros((1, 1, 128, 64), dtype=torch.float8_e4m3fn, device=dev)
    zb = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    with pytest.raises(ab.AttnError) as e:
        ab.attn_bwd_fp8(z, z, z, zb, z, lse, (1.0, 1.0, 1.0, 1.0), 1.0, False)
    assert e.value.status == ab.ATTN_ERR_UNSUPPORTED
    z = torch.zeros((1, 1, 128, 128), dtype=torch.float8_e4m3fn, device=dev)
    zb = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16, device=dev)
    for bad_ds in (0.0, float("inf")):
        with pytest.raises(ab.AttnError) as e:
            ab.attn_bwd_fp8(z, z, z, zb, z, lse, (1.0, 1.0, 1.0, 1.0), bad_ds, True)
        assert e.value.status == ab.ATTN_ERR_INVALID_ARG
