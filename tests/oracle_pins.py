"""Pins that tie the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes a loaded oracle library (so the same checks can
be run against deliberately broken copies of the oracle) and raises
AssertionError when the oracle disagrees with:

* central finite differences of its own forward (the gradient must be the
  derivative of the loss <dO, O>),
* closed forms (one key; zero queries; identical keys; two keys),
* invariants of softmax attention (rows of P sum to one, rows of dS sum to
  zero, shifting every key by one vector, permuting keys),
* PyTorch's own fp64 CPU attention and autograd (an independent library
  routine, used as a cross-check only),
* a pure-Python brute force over the full N x N matrices for N <= 8.

The sliding-window (banded causal) mask -- key j visible to query i when
i - W < j <= i -- has pins of its own: finite differences, the closed forms
W = 1 and W >= N, truncation to the window's keys, the brute force with the
band, and PyTorch with an explicit band mask.

Document masks (several sequences packed into one; a query sees keys of its
own document only, causally) are pinned by equality with separate causal
attention over each document, a single document being plain causal (bit for
bit), the brute force, and PyTorch with an explicit block-diagonal mask.

The method is exact attention as named by "Training Transformers and Hybrid
models on AMD Instinct MI300X Accelerators", section "Flash Attention"; the
pages print no worked example, so every pin is mathematical.
"""

from __future__ import annotations

import math

import numpy as np

import oracle


def _rand(rng, shape, std=1.0):
    return rng.standard_normal(shape) * std


def _fb(lib, q, k, v, do, causal, scale, window=0, doc=None):
    return oracle.attention_forward_backward(q, k, v, do, causal, scale, lib=lib,
                                             window=window, doc=doc)


def doc_map(lengths):
    """Document map of documents of the given lengths, packed in order:
    position i maps to the first position of its document."""
    out = []
    start = 0
    for n in lengths:
        out.extend([start] * n)
        start += n
    return np.array(out, dtype=np.int64)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, "%s: shape %s vs %s" % (what, a.shape, b.shape)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    ref = max(np.max(np.abs(b)) if b.size else 0.0, 1e-300)
    assert np.all(np.isfinite(a)), "%s: non-finite values" % what
    assert err <= rtol * ref + atol, "%s: max|err| %.3e > %.1e * %.3e + %.1e" % (
        what, err, rtol, ref, atol)


# --------------------------------------------------------------------------
# Finite differences: the backward is the derivative of the forward.
# --------------------------------------------------------------------------
def pin_finite_differences(lib):
    rng = np.random.default_rng(11)
    for causal in (False, True):
        for (N, d) in ((1, 2), (3, 2), (6, 4), (8, 3)):
            q, k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(4))
            scale = 0.7
            out = _fb(lib, q, k, v, do, causal, scale)

            def loss(q_, k_, v_):
                o, _ = oracle.attention_forward(q_, k_, v_, causal, scale, lib=lib)
                return float(np.sum(do * o))

            h = 1e-6
            for name, x, g in (("dQ", q, out["dQ"]), ("dK", k, out["dK"]),
                               ("dV", v, out["dV"])):
                num = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    xp = x.copy(); xp[idx] += h
                    xm = x.copy(); xm[idx] -= h
                    args_p = [q, k, v]; args_m = [q, k, v]
                    pos = {"dQ": 0, "dK": 1, "dV": 2}[name]
                    args_p[pos] = xp; args_m[pos] = xm
                    num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
                _close(g, num, rtol=1e-6, atol=1e-8,
                       what="finite differences %s N=%d d=%d causal=%s" % (name, N, d, causal))


# --------------------------------------------------------------------------
# Closed forms.
# --------------------------------------------------------------------------
def pin_single_key(lib):
    """N = 1: softmax over one key is 1, so O = V, L = s<q,k>, dV = dO, dQ = dK = 0."""
    rng = np.random.default_rng(12)
    for causal in (False, True):
        q, k, v, do = (_rand(rng, (2, 3, 1, 5)) for _ in range(4))
        s = 0.3
        out = _fb(lib, q, k, v, do, causal, s)
        _close(out["O"], v, 1e-15, what="N=1 O")
        _close(out["L"], s * np.sum(q * k, axis=-1), 1e-14, 1e-15, what="N=1 L")
        _close(out["dV"], do, 1e-15, what="N=1 dV")
        _close(out["dQ"], np.zeros_like(q), 0.0, 1e-15, what="N=1 dQ")
        _close(out["dK"], np.zeros_like(k), 0.0, 1e-15, what="N=1 dK")


def pin_zero_queries(lib):
    """Q = 0: every unmasked score is 0, so P is uniform over the unmasked keys.

    Non-causal: O_i = mean_j v_j and L_i = ln N.  Causal: O_i is the mean of
    v_0..v_i and L_i = ln(i + 1).
    """
    rng = np.random.default_rng(13)
    N, d = 37, 6
    q = np.zeros((1, 2, N, d))
    k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(3))
    out = _fb(lib, q, k, v, do, False, 0.4)
    _close(out["O"], np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape), 1e-13,
           what="Q=0 O")
    _close(out["L"], np.full((1, 2, N), math.log(N)), 1e-14, what="Q=0 L")
    out = _fb(lib, q, k, v, do, True, 0.4)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    _close(out["O"], prefix, 1e-13, what="Q=0 causal O")
    _close(out["L"], np.broadcast_to(np.log(np.arange(1, N + 1)), (1, 2, N)), 1e-14,
           what="Q=0 causal L")


def pin_identical_keys(lib):
    """All keys equal (non-causal): P is uniform and dS rows sum to zero, so
    O = mean(V), dQ = 0, and dV_j = mean_i-sum of dO / N for every j."""
    rng = np.random.default_rng(14)
    N, d = 19, 4
    q, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(3))
    k = np.broadcast_to(_rand(rng, (1, 1, 1, d)), (1, 1, N, d)).copy()
    out = _fb(lib, q, k, v, do, False, 0.9)
    _close(out["O"], np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape), 1e-13,
           what="equal keys O")
    _close(out["dQ"], np.zeros_like(q), 0.0, 1e-13, what="equal keys dQ")
    _close(out["dV"], np.broadcast_to(do.sum(axis=2, keepdims=True) / N, do.shape), 1e-13,
           what="equal keys dV")


def pin_two_keys_logistic(lib):
    """Two keys, d = 1, non-causal: P_i0 = sigmoid(s q_i (k_0 - k_1)).

    Then O_i = v_1 + sigmoid(a_i) (v_0 - v_1), and with a_i = s q_i (k_0 - k_1),
    dQ_i = s (k_0 - k_1) sigma'(a_i) (v_0 - v_1) dO_i.
    """
    q = np.array([0.5, -1.25, 2.0]).reshape(1, 1, 3, 1)
    k = np.array([0.75, -0.5, 0.0]).reshape(1, 1, 3, 1)
    # only the first two keys exist: N must match, so build N=2 queries twice
    for i in range(3):
        qi = q[:, :, i:i + 1, :].repeat(2, axis=2)
        kk = k[:, :, :2, :]
        v = np.array([3.0, -1.0]).reshape(1, 1, 2, 1)
        do = np.array([0.25, 0.0]).reshape(1, 1, 2, 1)
        s = 1.5
        out = _fb(lib, qi, kk, v, do, False, s)
        a = s * q[0, 0, i, 0] * (k[0, 0, 0, 0] - k[0, 0, 1, 0])
        sig = 1.0 / (1.0 + math.exp(-a))
        o_expect = v[0, 0, 1, 0] + sig * (v[0, 0, 0, 0] - v[0, 0, 1, 0])
        assert abs(out["O"][0, 0, 0, 0] - o_expect) <= 1e-14, "two-key O"
        dq_expect = (s * (k[0, 0, 0, 0] - k[0, 0, 1, 0]) * sig * (1 - sig)
                     * (v[0, 0, 0, 0] - v[0, 0, 1, 0]) * do[0, 0, 0, 0])
        assert abs(out["dQ"][0, 0, 0, 0] - dq_expect) <= 1e-14, "two-key dQ"
        lse = max(s * q[0, 0, i, 0] * k[0, 0, 0, 0], s * q[0, 0, i, 0] * k[0, 0, 1, 0])
        lse += math.log(math.exp(s * q[0, 0, i, 0] * k[0, 0, 0, 0] - lse)
                        + math.exp(s * q[0, 0, i, 0] * k[0, 0, 1, 0] - lse))
        assert abs(out["L"][0, 0, 0] - lse) <= 1e-14, "two-key L"


# --------------------------------------------------------------------------
# Invariants.
# --------------------------------------------------------------------------
def pin_invariants(lib):
    """Rows of P sum to one and rows of dS sum to zero, seen through outputs.

    * sum_j dV_j = sum_i (sum_j P_ij) dO_i = sum_i dO_i.
    * sum_j dK_j = s sum_i q_i sum_j dS_ij = 0.
    * adding one vector c to every key leaves O, dQ, dK, dV unchanged and moves
      L_i by s <q_i, c> (each score row moves by a constant).
    * O_i is a convex combination of the value rows it can see.
    * scaling V scales O and leaves dV unchanged (dV = P^T dO).
    """
    rng = np.random.default_rng(15)
    for causal in (False, True):
        B, H, N, d = 2, 2, 45, 7
        q, k, v, do = (_rand(rng, (B, H, N, d)) for _ in range(4))
        s = 0.45
        out = _fb(lib, q, k, v, do, causal, s)
        _close(out["dV"].sum(axis=2), do.sum(axis=2), 1e-12, what="sum dV = sum dO")
        _close(out["dK"].sum(axis=2), np.zeros((B, H, d)), 0.0,
               1e-12 * np.abs(out["dK"]).max(), what="sum dK = 0")
        c = _rand(rng, (1, 1, 1, d))
        out2 = _fb(lib, q, k + c, v, do, causal, s)
        for name in ("O", "dQ", "dK", "dV"):
            _close(out2[name], out[name], 1e-11, what="key shift %s" % name)
        _close(out2["L"], out["L"] + s * np.sum(q * c, axis=-1), 1e-12,
               what="key shift L")
        if causal:
            lo = np.minimum.accumulate(v, axis=2)
            hi = np.maximum.accumulate(v, axis=2)
        else:
            lo = np.broadcast_to(v.min(axis=2, keepdims=True), v.shape)
            hi = np.broadcast_to(v.max(axis=2, keepdims=True), v.shape)
        assert np.all(out["O"] >= lo - 1e-12) and np.all(out["O"] <= hi + 1e-12), "convexity"
        out3 = _fb(lib, q, k, 2.5 * v, do, causal, s)
        _close(out3["O"], 2.5 * out["O"], 1e-13, what="V scaling O")
        _close(out3["dV"], out["dV"], 1e-13, what="V scaling dV")
        _close(out["D"], np.sum(do * out["O"], axis=-1), 1e-13, what="D = rowsum(dO*O)")


def pin_permutation(lib):
    """Non-causal attention is equivariant in the queries and invariant to a
    joint permutation of the keys and values."""
    rng = np.random.default_rng(16)
    N, d = 23, 5
    q, k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(4))
    out = _fb(lib, q, k, v, do, False, 0.6)
    pk = rng.permutation(N)
    pq = rng.permutation(N)
    out2 = _fb(lib, q[:, :, pq], k[:, :, pk], v[:, :, pk], do[:, :, pq], False, 0.6)
    for name in ("O", "dQ"):
        _close(out2[name], out[name][:, :, pq], 1e-12, what="perm %s" % name)
    _close(out2["L"], out["L"][:, :, pq], 1e-12, what="perm L")
    for name in ("dK", "dV"):
        _close(out2[name], out[name][:, :, pk], 1e-12, what="perm %s" % name)


# --------------------------------------------------------------------------
# Brute force over the full matrices, pure Python loops, tiny N.
# --------------------------------------------------------------------------
def _brute(q, k, v, do, causal, s, window=0, doc=None):
    N, d = len(q), len(q[0])

    def visible(i, j):
        if not causal:
            return True
        same_doc = doc is None or doc[i] == doc[j]
        return j <= i and (window == 0 or i - j < window) and same_doc

    S = [[(s * sum(q[i][c] * k[j][c] for c in range(d)) if visible(i, j)
           else -math.inf) for j in range(N)] for i in range(N)]
    L = []
    for i in range(N):
        m = max(S[i])
        L.append(m + math.log(sum(math.exp(x - m) for x in S[i])))
    P = [[math.exp(S[i][j] - L[i]) for j in range(N)] for i in range(N)]
    O = [[sum(P[i][j] * v[j][c] for j in range(N)) for c in range(d)] for i in range(N)]
    dP = [[sum(do[i][c] * v[j][c] for c in range(d)) for j in range(N)] for i in range(N)]
    D = [sum(do[i][c] * O[i][c] for c in range(d)) for i in range(N)]
    dS = [[P[i][j] * (dP[i][j] - D[i]) for j in range(N)] for i in range(N)]
    dQ = [[s * sum(dS[i][j] * k[j][c] for j in range(N)) for c in range(d)] for i in range(N)]
    dK = [[s * sum(dS[i][j] * q[i][c] for i in range(N)) for c in range(d)] for j in range(N)]
    dV = [[sum(P[i][j] * do[i][c] for i in range(N)) for c in range(d)] for j in range(N)]
    rowsum_P = [sum(P[i]) for i in range(N)]
    rowsum_dS = [sum(dS[i]) for i in range(N)]
    return dict(O=O, L=L, D=D, dQ=dQ, dK=dK, dV=dV, rowsum_P=rowsum_P, rowsum_dS=rowsum_dS)


def pin_brute_force(lib):
    rng = np.random.default_rng(17)
    for causal in (False, True):
        for N, d in ((2, 1), (5, 3), (8, 4)):
            q, k, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(4))
            s = 0.8
            out = _fb(lib, q, k, v, do, causal, s)
            ref = _brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                         do[0, 0].tolist(), causal, s)
            _close(ref["rowsum_P"], np.ones(N), 1e-14, what="brute rowsum P")
            assert max(abs(x) for x in ref["rowsum_dS"]) < 1e-12, "brute rowsum dS"
            for name in ("O", "dQ", "dK", "dV"):
                _close(out[name][0, 0], np.array(ref[name]), 1e-12,
                       what="brute %s N=%d causal=%s" % (name, N, causal))
            for name in ("L", "D"):
                _close(out[name][0, 0], np.array(ref[name]), 1e-12,
                       what="brute %s" % name)


# --------------------------------------------------------------------------
# Independent library cross-check: PyTorch fp64 CPU attention + autograd.
# --------------------------------------------------------------------------
def _sdpa_fp64(torch, q, k, v, **kw):
    """PyTorch's scaled_dot_product_attention on its plain math backend
    (matmul and softmax composed in the inputs' fp64), not a fused kernel."""
    from torch.nn.attention import SDPBackend, sdpa_kernel

    with sdpa_kernel(SDPBackend.MATH):
        return torch.nn.functional.scaled_dot_product_attention(q, k, v, **kw)


def pin_torch_fp64(lib):
    import torch

    rng = np.random.default_rng(18)
    for causal in (False, True):
        for (B, H, N, d) in ((1, 2, 64, 16), (2, 1, 131, 8), (1, 1, 300, 32)):
            q, k, v, do = (_rand(rng, (B, H, N, d)) for _ in range(4))
            s = 1.0 / math.sqrt(d)
            out = _fb(lib, q, k, v, do, causal, s)
            tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True)
                          for x in (q, k, v))
            to = _sdpa_fp64(torch, tq, tk, tv, is_causal=causal, scale=s)
            to.backward(torch.tensor(do, dtype=torch.float64))
            scores = (tq.detach() @ tk.detach().transpose(-1, -2)) * s
            if causal:
                mask = torch.ones(N, N, dtype=torch.bool).triu(1)
                scores = scores.masked_fill(mask, float("-inf"))
            tl = torch.logsumexp(scores, dim=-1)
            _close(out["O"], to.detach().numpy(), 1e-11, what="torch O")
            _close(out["L"], tl.numpy(), 1e-12, what="torch L")
            _close(out["dQ"], tq.grad.numpy(), 1e-10, what="torch dQ")
            _close(out["dK"], tk.grad.numpy(), 1e-10, what="torch dK")
            _close(out["dV"], tv.grad.numpy(), 1e-10, what="torch dV")




def pin_row_sampler_matches_full(lib):
    """The row sampler evaluates the same definition as the full oracle: its
    rows equal the full result's rows bit for bit (same arithmetic order),
    under every mask it takes -- none, causal, a sliding window, documents,
    and documents with a window.  The large-size GPU tests of the mask
    variants rely on the sampler in those modes."""
    rng = np.random.default_rng(19)
    N, d = 57, 6
    docs = doc_map([9, 1, 20, 27])  # a one-position document, documents across the rows
    cases = [(False, 0, None), (True, 0, None), (True, 5, None), (True, 1, None),
             (True, 0, docs), (True, 7, docs)]
    for causal, window, doc in cases:
        q, k, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(4))
        full = _fb(lib, q, k, v, do, causal, 0.35, window=window,
                   doc=None if doc is None else doc[None, :])
        qr, kr = [0, 5, 9, 10, 56, 31], [56, 0, 9, 13, 30]
        what = "causal=%s window=%d doc=%s" % (causal, window, doc is not None)
        rows = oracle.attention_head_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, 0.35,
                                          qr, kr, lib=lib, window=window, doc=doc)
        for name in ("O", "dQ"):
            assert np.array_equal(rows[name], full[name][0, 0][qr]), (name, what)
        assert np.array_equal(rows["L"], full["L"][0, 0][qr]), what
        for name in ("dK", "dV"):
            assert np.array_equal(rows[name], full[name][0, 0][kr]), (name, what)
        # query rows only (no key rows): each row is evaluated on its own
        qonly = oracle.attention_head_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, 0.35,
                                           qr, [], lib=lib, window=window, doc=doc)
        for name in ("O", "dQ"):
            assert np.array_equal(qonly[name], full[name][0, 0][qr]), (name, what)
        assert np.array_equal(qonly["L"], full["L"][0, 0][qr]), what


# --------------------------------------------------------------------------
# Sliding window (banded causal mask).
# --------------------------------------------------------------------------
def pin_window_finite_differences(lib):
    rng = np.random.default_rng(21)
    for (N, d, W) in ((5, 2, 2), (7, 3, 3), (6, 2, 1)):
        q, k, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(4))
        scale = 0.9
        out = _fb(lib, q, k, v, do, True, scale, window=W)

        def loss(q_, k_, v_):
            o, _ = oracle.attention_forward(q_, k_, v_, True, scale, lib=lib, window=W)
            return float(np.sum(do * o))

        h = 1e-6
        for pos, name in enumerate(("dQ", "dK", "dV")):
            x = (q, k, v)[pos]
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy(); xp[idx] += h
                xm = x.copy(); xm[idx] -= h
                args_p = [q, k, v]; args_m = [q, k, v]
                args_p[pos] = xp; args_m[pos] = xm
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            _close(out[name], num, rtol=1e-6, atol=1e-8,
                   what="window finite differences %s N=%d W=%d" % (name, N, W))


def pin_window_closed_forms(lib):
    """W >= N is the plain causal mask (bit for bit); W = 1 leaves each query
    only itself: P = 1, so O = V, L_i = s<q_i,k_i>, dV = dO and dS = 0, hence
    dQ = dK = 0 exactly."""
    rng = np.random.default_rng(22)
    N, d, s = 19, 4, 0.45
    q, k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(4))
    causal = _fb(lib, q, k, v, do, True, s)
    for W in (N, N + 5, 1000):
        wide = _fb(lib, q, k, v, do, True, s, window=W)
        for name in causal:
            assert np.array_equal(wide[name], causal[name]), "W=%d %s" % (W, name)
    one = _fb(lib, q, k, v, do, True, s, window=1)
    assert np.array_equal(one["O"], v), "W=1: O = V"
    _close(one["L"], s * np.sum(q * k, axis=-1), 1e-14, what="W=1: L")
    assert np.array_equal(one["dV"], do), "W=1: dV = dO"
    assert not np.any(one["dQ"]) and not np.any(one["dK"]), "W=1: dQ = dK = 0"


def pin_window_truncation(lib):
    """Query i under a window W attends exactly to keys i-W+1 .. i: its O, L
    and dQ equal those of unmasked attention of q_i over that slice alone."""
    rng = np.random.default_rng(23)
    N, d, W, s = 40, 5, 7, 0.5
    q, k, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(4))
    out = _fb(lib, q, k, v, do, True, s, window=W)
    for i in (0, 3, 6, 7, 20, 39):
        lo = max(0, i - W + 1)
        n = i + 1 - lo
        qi = np.repeat(q[:, :, i:i + 1], n, axis=2)
        doi = np.repeat(do[:, :, i:i + 1], n, axis=2)
        part = _fb(lib, qi, k[:, :, lo:i + 1], v[:, :, lo:i + 1], doi, False, s)
        _close(out["O"][0, 0, i], part["O"][0, 0, 0], 1e-13, what="trunc O row %d" % i)
        _close(out["L"][0, 0, i], part["L"][0, 0, 0], 1e-13, what="trunc L row %d" % i)
        _close(out["dQ"][0, 0, i], part["dQ"][0, 0, 0], 1e-12, what="trunc dQ row %d" % i)


def pin_window_brute_force(lib):
    rng = np.random.default_rng(24)
    for N, d, W in ((5, 2, 2), (8, 3, 3), (8, 2, 5)):
        q, k, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(4))
        s = 0.8
        out = _fb(lib, q, k, v, do, True, s, window=W)
        ref = _brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                     do[0, 0].tolist(), True, s, window=W)
        for name in ("O", "dQ", "dK", "dV", "L", "D"):
            _close(out[name][0, 0], np.array(ref[name]), 1e-12,
                   what="window brute %s N=%d W=%d" % (name, N, W))


def pin_window_torch_fp64(lib):
    import torch

    rng = np.random.default_rng(25)
    for (N, d, W) in ((64, 16, 16), (131, 8, 50), (300, 32, 129)):
        q, k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(4))
        s = 1.0 / math.sqrt(d)
        out = _fb(lib, q, k, v, do, True, s, window=W)
        i = torch.arange(N).view(N, 1)
        j = torch.arange(N).view(1, N)
        band = (j <= i) & (i - j < W)  # True = attend
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True)
                      for x in (q, k, v))
        to = _sdpa_fp64(torch, tq, tk, tv, attn_mask=band, scale=s)
        to.backward(torch.tensor(do, dtype=torch.float64))
        _close(out["O"], to.detach().numpy(), 1e-11, what="window torch O")
        _close(out["dQ"], tq.grad.numpy(), 1e-10, what="window torch dQ")
        _close(out["dK"], tk.grad.numpy(), 1e-10, what="window torch dK")
        _close(out["dV"], tv.grad.numpy(), 1e-10, what="window torch dV")


# --------------------------------------------------------------------------
# Document masks (packed sequences).
# --------------------------------------------------------------------------
def pin_doc_separate_sequences(lib):
    """Packed documents give exactly what each document gives on its own under
    the plain causal mask: O, L, D, dQ, dK, dV, row by row."""
    rng = np.random.default_rng(26)
    for lengths in ((5, 1, 9, 3), (17,), (1, 1, 1), (12, 30, 7)):
        N, d, s = sum(lengths), 4, 0.6
        q, k, v, do = (_rand(rng, (2, 2, N, d)) for _ in range(4))
        dm = np.stack([doc_map(lengths), doc_map(lengths)])
        packed = _fb(lib, q, k, v, do, True, s, doc=dm)
        start = 0
        for n in lengths:
            sl = slice(start, start + n)
            alone = _fb(lib, q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], True, s)
            for name in ("O", "dQ", "dK", "dV"):
                _close(packed[name][:, :, sl], alone[name], 1e-13,
                       what="doc %s lengths=%s" % (name, lengths))
            for name in ("L", "D"):
                _close(packed[name][:, :, sl], alone[name], 1e-13, what="doc %s" % name)
            start += n


def pin_doc_single_document_is_causal(lib):
    rng = np.random.default_rng(27)
    N, d, s = 33, 3, 0.7
    q, k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(4))
    one = _fb(lib, q, k, v, do, True, s, doc=np.zeros((1, N), dtype=np.int64))
    causal = _fb(lib, q, k, v, do, True, s)
    for name in causal:
        assert np.array_equal(one[name], causal[name]), name


def pin_doc_brute_force(lib):
    rng = np.random.default_rng(28)
    for lengths, W in (((3, 5), 0), ((2, 2, 4), 0), ((6, 2), 3), ((1, 7), 2)):
        N, d, s = sum(lengths), 3, 0.8
        q, k, v, do = (_rand(rng, (1, 1, N, d)) for _ in range(4))
        dm = doc_map(lengths)
        out = _fb(lib, q, k, v, do, True, s, window=W, doc=dm[None])
        ref = _brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                     do[0, 0].tolist(), True, s, window=W, doc=dm.tolist())
        for name in ("O", "dQ", "dK", "dV", "L", "D"):
            _close(out[name][0, 0], np.array(ref[name]), 1e-12,
                   what="doc brute %s lengths=%s W=%d" % (name, lengths, W))


def pin_doc_torch_fp64(lib):
    import torch

    rng = np.random.default_rng(29)
    for lengths, W in (((40, 24), 0), ((100, 1, 30), 0), ((70, 90, 140), 50)):
        N, d = sum(lengths), 16
        q, k, v, do = (_rand(rng, (1, 2, N, d)) for _ in range(4))
        s = 1.0 / math.sqrt(d)
        dm = doc_map(lengths)
        out = _fb(lib, q, k, v, do, True, s, window=W, doc=dm[None])
        i = torch.arange(N).view(N, 1)
        j = torch.arange(N).view(1, N)
        dt = torch.tensor(dm)
        allowed = (j <= i) & (dt.view(N, 1) == dt.view(1, N))
        if W:
            allowed &= i - j < W
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True)
                      for x in (q, k, v))
        to = _sdpa_fp64(torch, tq, tk, tv, attn_mask=allowed, scale=s)
        to.backward(torch.tensor(do, dtype=torch.float64))
        _close(out["O"], to.detach().numpy(), 1e-11, what="doc torch O")
        _close(out["dQ"], tq.grad.numpy(), 1e-10, what="doc torch dQ")
        _close(out["dK"], tk.grad.numpy(), 1e-10, what="doc torch dK")
        _close(out["dV"], tv.grad.numpy(), 1e-10, what="doc torch dV")


# --------------------------------------------------------------------------
# The E4M3 decoder of the fp8 path.
# --------------------------------------------------------------------------
def pin_e4m3_decoder(lib):
    """The decoder against values the format's definition fixes by hand
    (1, the largest finite 448, the smallest normal 2^-6 and subnormal 2^-9,
    signs, NaN), against brute force over sign/exponent/mantissa, and against
    PyTorch's own float8_e4m3fn -> float64 conversion of all 256 codes."""
    from oracle import fp8

    fixed = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0, 0x08: 2.0 ** -6,
             0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x40: 2.0, 0x39: 1.125, 0x30: 0.5,
             0x3F: 1.875, 0x77: 240.0}
    for code, val in fixed.items():
        assert fp8.e4m3_to_f64(code) == val, hex(code)
    assert np.isnan(fp8.e4m3_to_f64(0x7F)) and np.isnan(fp8.e4m3_to_f64(0xFF))
    codes = np.arange(256)
    got = fp8.e4m3_to_f64(codes)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(got[c])
            continue
        mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert got[c] == (-mag if s else mag), hex(c)
    try:
        import torch
    except ImportError:  # the cross-check needs PyTorch; the other checks stand
        return
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    ref = ref.numpy()
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


def pin_rounding_budget_brute_force(lib):
    """The rounding-budget sums of the 8-bit backward against full N x N
    matrices built in numpy (P, dP, dS written out from the definition)."""
    rng = np.random.default_rng(29)
    for causal in (False, True):
        B, H, N, d = 1, 2, 9, 4
        q, k, v, do = (_rand(rng, (B, H, N, d)) for _ in range(4))
        s = 0.41
        ref = _fb(lib, q, k, v, do, causal, s)
        got = oracle.backward_rounding_budget(q, k, v, do, causal, s, ref["L"], ref["D"],
                                              lib=lib)
        for h in range(H):
            S = s * q[0, h] @ k[0, h].T
            if causal:
                S = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            P = np.exp(S - m)
            P /= P.sum(axis=1, keepdims=True)
            O = P @ v[0, h]
            Dv = np.sum(do[0, h] * O, axis=1)
            dS = P * (do[0, h] @ v[0, h].T - Dv[:, None])
            _close(got["vP"][0, h], (P ** 2).T @ do[0, h] ** 2, 1e-12, what="budget vP")
            _close(got["vK"][0, h], (dS ** 2).T @ q[0, h] ** 2, 1e-12, what="budget vK")
            _close(got["vQ"][0, h], (dS ** 2) @ k[0, h] ** 2, 1e-12, what="budget vQ")
            vis = np.tril(np.ones((N, N))) if causal else np.ones((N, N))
            assert np.array_equal(got["nvis"][0, h], vis.sum(axis=0))
            _close(got["dsmax"][0, h], np.abs(dS).max(), 1e-12, what="budget dsmax")


ALL_PINS = [
    pin_finite_differences,
    pin_single_key,
    pin_zero_queries,
    pin_identical_keys,
    pin_two_keys_logistic,
    pin_invariants,
    pin_permutation,
    pin_brute_force,
    pin_torch_fp64,
    pin_row_sampler_matches_full,
    pin_window_finite_differences,
    pin_window_closed_forms,
    pin_window_truncation,
    pin_window_brute_force,
    pin_window_torch_fp64,
    pin_doc_separate_sequences,
    pin_doc_single_document_is_causal,
    pin_doc_brute_force,
    pin_doc_torch_fp64,
    pin_e4m3_decoder,
    pin_rounding_budget_brute_force,
]
