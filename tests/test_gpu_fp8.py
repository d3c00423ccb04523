"""The e4m3 (fp8) forward on the GPU against the fp64 oracle.

The fp8 entry point takes E4M3 bytes and one descale factor per tensor; what
it computes is exact attention of the values those stand for, so the oracle
decodes them (``oracle.fp8``) and runs its exact forward on them.  The only
rounding the kernel adds beyond the bf16 path is that of the probabilities
to e4m3 for the P V contraction; the tolerance follows from it:

* L (natural-log log-sum-exp) uses the unrounded fp32 probabilities:
  |L_gpu - L| <= 2e-3 (fp32 accumulation of exact 8-bit products).
* O: round-to-nearest e4m3 has a relative error |d| <= 2^-4 (three mantissa
  bits), and probabilities below e4m3's normal range (p < 2^-14 of the row
  maximum, as the kernel scales them) an absolute error <= 2^-18.  Treating
  the roundings as independent and uniform, element (i, c) of O has the
  standard deviation
      sigma_ic^2 = (2^-4)^2/3 sum_j p_ij^2 v_jc^2 + (2^-18)^2/3 sum_j v_jc^2
  (sums over the keys row i sees).  The oracle supplies the first sum with
  its own forward at twice the scale on V o V: sum_j p_ij^2 v_jc^2 =
  O'_ic exp(L'_i - 2 L_i).  Every element must satisfy
      |O_gpu - O| <= 7 sigma + 2^-8 |O| (the bf16 output) + 1e-5 max|O|,
  and the root-mean-square error over the tensor must stay within 1.5x the
  predicted one.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import (WORKLOADS, make_inputs_fp8, make_tensor,
                                                       quantize_e4m3)

pytestmark = pytest.mark.gpu

L_ATOL = 2e-3


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


def run_gpu(q8, k8, v8, descales, causal, scale):
    dev = torch.device("cuda", 0)
    o, lse = ab.attn_fwd_fp8(q8.to(dev), k8.to(dev), v8.to(dev), descales, causal, scale)
    torch.cuda.synchronize()
    st, word = ab.attn_device_error_word()
    assert st == ab.ATTN_OK, "device error %d word 0x%08x" % (st, word)
    return o.cpu().to(torch.float64).numpy(), lse.cpu().to(torch.float64).numpy()


def check(q8, qd, k8, kd, v8, vd, causal, scale, what):
    o_gpu, l_gpu = run_gpu(q8, k8, v8, (qd, kd, vd), causal, scale)
    q, k, v = fp8.dequantize(q8, qd), fp8.dequantize(k8, kd), fp8.dequantize(v8, vd)
    o_ref, l_ref = oracle.attention_forward(q, k, v, causal, scale)
    o2, l2 = oracle.attention_forward(q, k, v * v, causal, 2 * scale)
    sum_p2v2 = o2 * np.exp(l2 - 2 * l_ref)[..., None]
    # sum of v^2 over the keys each row sees (all keys, or a prefix)
    vv = v * v
    sum_v2 = np.cumsum(vv, axis=2) if causal else np.broadcast_to(vv.sum(2, keepdims=True),
                                                                   vv.shape)
    var = (2.0 ** -4) ** 2 / 3 * sum_p2v2 + (2.0 ** -18) ** 2 / 3 * sum_v2
    sigma = np.sqrt(np.maximum(var, 0.0))
    err = np.abs(o_gpu - o_ref)
    omax = float(np.max(np.abs(o_ref))) if o_ref.size else 0.0
    bound = 7 * sigma + 2.0 ** -8 * np.abs(o_ref) + 1e-5 * omax
    assert np.all(np.isfinite(o_gpu)), what
    worst = float(np.max(err / bound)) if err.size else 0.0
    lerr = float(np.max(np.abs(l_gpu - l_ref))) if l_ref.size else 0.0
    rms, rms_pred = (float(np.sqrt(np.mean(err ** 2))),
                     float(np.sqrt(np.mean(var + (2.0 ** -9 * o_ref) ** 2)))) if err.size \
        else (0.0, 0.0)
    rel = float(np.max(err) / omax) if omax > 0 else 0.0
    msg = ("%s: worst err/bound %.3f, rms %.3e (predicted %.3e), max|err|/max|O| %.3e, "
           "L abs %.2e" % (what, worst, rms, rms_pred, rel, lerr))
    assert worst <= 1.0, msg
    assert rms <= 1.5 * rms_pred + 1e-7, msg
    assert lerr <= L_ATOL, msg
    return rel


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("N", [1, 7, 100, 128, 129, 300, 513])
def test_fp8_ragged_lengths(N, causal):
    B, H, d = 1, 3, 128
    seed = 3000 + N * 2 + int(causal)
    q, k, v = (make_tensor((B, H, N, d), seed + 7919 * i) for i in range(3))
    (q8, qd), (k8, kd), (v8, vd) = quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v)
    check(q8, qd, k8, kd, v8, vd, causal, 1 / math.sqrt(d), "N=%d causal=%s" % (N, causal))


@pytest.mark.parametrize("qscale", [1.0, 4.0])
def test_fp8_sharp_and_flat_softmax(qscale):
    """Peaked rows (large logits: one probability near 1 carries the e4m3
    error of one term) and flat ones."""
    B, H, N, d = 1, 4, 640, 128
    q = make_tensor((B, H, N, d), 61, std=qscale)
    k, v = (make_tensor((B, H, N, d), 62 + i) for i in range(2))
    (q8, qd), (k8, kd), (v8, vd) = quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v)
    for causal in (False, True):
        check(q8, qd, k8, kd, v8, vd, causal, 1 / math.sqrt(d),
              "q x%g causal=%s" % (qscale, causal))


@pytest.mark.parametrize("name", ["b1h32n4096d128_causal", "b4h16n8192d128",
                                  "b1h16n16384d128_causal"])
def test_fp8_workloads_full_tensors(name):
    """The three d = 128 named workloads, quantised to e4m3 per tensor, at full
    size over the whole O and L."""
    w = WORKLOADS[name]
    (q8, qd), (k8, kd), (v8, vd), _ = make_inputs_fp8(w)
    check(q8, qd, k8, kd, v8, vd, w.causal, w.scale, name)


def test_fp8_argument_checks():
    dev = torch.device("cuda", 0)
    z = torch.zeros((1, 1, 128, 64), dtype=torch.float8_e4m3fn, device=dev)
    with pytest.raises(ab.AttnError) as e:  # head dim 64 is not offered
        ab.attn_fwd_fp8(z, z, z, (1.0, 1.0, 1.0), False)
    assert e.value.status == ab.ATTN_ERR_UNSUPPORTED
    z = torch.zeros((1, 1, 128, 128), dtype=torch.float8_e4m3fn, device=dev)
    for bad in ((0.0, 1.0, 1.0), (1.0, float("nan"), 1.0), (1.0, 1.0, -2.0)):
        with pytest.raises(ab.AttnError) as e:
            ab.attn_fwd_fp8(z, z, z, bad, False)
        assert e.value.status == ab.ATTN_ERR_INVALID_ARG
    e0 = torch.zeros((1, 1, 0, 128), dtype=torch.float8_e4m3fn, device=dev)
    o, lse = ab.attn_fwd_fp8(e0, e0, e0, (1.0, 1.0, 1.0), True)
    assert o.shape == (1, 1, 0, 128) and lse.shape == (1, 1, 0)
