"""Document masks (several sequences packed into one) on the GPU against the
fp64 oracle: a query sees keys of its own document only, causally, i.e.
doc[i] <= j <= i with doc[i] the first position of i's document.

Random packings with documents shorter than, equal to and longer than a
128-row tile, different packings per batch element, documents combined with
a sliding window, one document (bit-equal to the causal mask), and sampled
rows at a long-sequence size.
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


def doc_map(lengths):
    out, start = [], 0
    for n in lengths:
        out.extend([start] * n)
        start += n
    return np.array(out, dtype=np.int64)


def random_lengths(rng, N, lo, hi):
    lengths = []
    while sum(lengths) < N:
        lengths.append(int(min(rng.integers(lo, hi + 1), N - sum(lengths))))
    return lengths


METHODS = {"reduce": ab.ATTN_DQ_REDUCE, "separate": ab.ATTN_DQ_SEPARATE}


def run(q, k, v, do, scale, window, docs, dq_method=ab.ATTN_DQ_AUTO):
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    dmap = torch.from_numpy(docs.astype(np.int32)).to(dev)
    o, lse = ab.attn_fwd(qd, kd, vd, True, scale, window=window, doc=dmap)
    dq, dk, dv = ab.attn_bwd(qd, kd, vd, o, dod, lse, True, scale, window=window, doc=dmap,
                             dq_method=dq_method)
    torch.cuda.synchronize()
    return dict(O=o, L=lse, dQ=dq, dK=dk, dV=dv)


def check(gpu, ref, what):
    errs = {n: rel_err(gpu[n], ref[n]) for n in ("O", "dQ", "dK", "dV")}
    lerr = float(np.max(np.abs(f64(gpu["L"]) - ref["L"])))
    msg = "%s: %s L %.2e" % (what, {k: "%.2e" % v for k, v in errs.items()}, lerr)
    assert all(e <= TOL for e in errs.values()), msg
    assert lerr <= L_ATOL, msg


@pytest.mark.parametrize("method", sorted(METHODS))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,lo,hi,window", [(129, 1, 40, 0), (300, 20, 200, 0),
                                            (700, 100, 400, 0), (1000, 1, 700, 0),
                                            (640, 128, 128, 0), (900, 50, 500, 96),
                                            (513, 200, 513, 300)])
def test_documents_full_tensors(N, lo, hi, window, d, method):
    rng = np.random.default_rng(N * 31 + lo + hi + window + d)
    B, H = 2, 2
    docs = np.stack([doc_map(random_lengths(rng, N, lo, hi)) for _ in range(B)])
    seed = 7000 + N + d + window
    q, k, v, do = (make_tensor((B, H, N, d), seed + 7919 * i) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_forward_backward(q, k, v, do, True, scale, window=window, doc=docs)
    gpu = run(q, k, v, do, scale, window, docs, METHODS[method])
    check(gpu, ref, "N=%d docs %d..%d W=%d d=%d dq=%s" % (N, lo, hi, window, d, method))


def test_one_document_is_causal():
    B, H, N, d = 1, 2, 400, 64
    q, k, v, do = (make_tensor((B, H, N, d), 61 + i) for i in range(4))
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    zero = torch.zeros((B, N), dtype=torch.int32, device=dev)
    o1, l1 = ab.attn_fwd(qd, kd, vd, True)
    o2, l2 = ab.attn_fwd(qd, kd, vd, True, doc=zero)
    g1 = ab.attn_bwd(qd, kd, vd, o1, dod, l1, True)
    g2 = ab.attn_bwd(qd, kd, vd, o1, dod, l1, True, doc=zero)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert rel_err(g2[0], f64(g1[0])) <= 2e-3


@pytest.mark.parametrize("method", sorted(METHODS))
def test_documents_long_sequence_sampled(method):
    """N = 16384, d = 128, documents of 300 to 5000 positions: sampled rows."""
    B, H, N, d = 1, 4, 16384, 128
    rng = np.random.default_rng(8)
    docs = doc_map(random_lengths(rng, N, 300, 5000))[None]
    q, k, v, do = (make_tensor((B, H, N, d), 950 + i) for i in range(4))
    scale = 1.0 / math.sqrt(d)
    gpu = run(q, k, v, do, scale, 0, docs, METHODS[method])
    starts = sorted(set(docs[0].tolist()))
    for h in (0, H - 1):
        rows = sorted(set([0, 1, 127, 128, N - 1] + starts[:6] + [max(s - 1, 0) for s in starts[:6]]
                          + rng.choice(N, 30, replace=False).tolist()))
        ref = oracle.attention_head_rows(q[0, h], k[0, h], v[0, h], do[0, h], True, scale,
                                         rows, rows, doc=docs[0])
        errs = {"O": rel_err(gpu["O"][0, h][rows], ref["O"]),
                "dQ": rel_err(gpu["dQ"][0, h][rows], ref["dQ"]),
                "dK": rel_err(gpu["dK"][0, h][rows], ref["dK"]),
                "dV": rel_err(gpu["dV"][0, h][rows], ref["dV"])}
        lerr = float(np.max(np.abs(f64(gpu["L"][0, h][rows]) - ref["L"])))
        msg = "head %d: %s L %.2e" % (h, errs, lerr)
        assert all(e <= TOL for e in errs.values()), msg
        assert lerr <= L_ATOL, msg


def test_documents_many_batch_elements_forward():
    """65 batch elements of N = 16384, each with its own packing (4160
    query-tile pairs, one forward CTA each): sampled rows of O and L in the
    first, a middle and the last batch element."""
    B, H, N, d = 65, 1, 16384, 64
    rng = np.random.default_rng(65)
    docs = np.stack([doc_map(random_lengths(rng, N, 200, 3000)) for _ in range(B)])
    q, k, v = (make_tensor((B, H, N, d), 6500 + i) for i in range(3))
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", 0)
    dmap = torch.from_numpy(docs.astype(np.int32)).to(dev)
    o, lse = ab.attn_fwd(q.to(dev), k.to(dev), v.to(dev), True, scale, doc=dmap)
    torch.cuda.synchronize()
    for b in (0, B // 2, B - 1):
        starts = sorted(set(docs[b].tolist()))
        rows = sorted(set([0, 127, 128, N - 1] + starts[:4] + [max(s - 1, 0) for s in starts[:4]]
                          + rng.choice(N, 16, replace=False).tolist()))
        ref = oracle.attention_head_rows(q[b, 0], k[b, 0], v[b, 0], q[b, 0], True, scale,
                                         rows, [0], doc=docs[b])
        err = rel_err(o[b, 0][rows], ref["O"])
        lerr = float(np.max(np.abs(f64(lse[b, 0][rows]) - ref["L"])))
        assert err <= TOL and lerr <= L_ATOL, "batch element %d: O %.2e L %.2e" % (b, err, lerr)
