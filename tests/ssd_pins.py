"""Pins that tie the fp64 Mamba-2 (SSD) oracle to facts other than itself.

Each ``pin_*`` takes a loaded oracle library (so the same checks run against
deliberately broken copies of it) and raises AssertionError on a mismatch
with:

* central finite differences of the oracle's own forward (every gradient is
  the derivative of the loss <dy, y>: x, dt, A, B, C, D);
* the dual form of the same layer, written independently here: with
  cs_t = sum_{r <= t} dt_r, y_t = sum_{s <= t} (C_t . B_s) dt_s
  exp(A (cs_t - cs_s)) x_s + D x_t (a masked, decayed attention-like
  matrix), and its analytic gradients;
* closed forms: a single step; A = 0 (no decay: cumulative sums); a decay
  that underflows to zero (no memory: y_t = dt_t (C_t . B_t) x_t + D x_t);
* the sharing of B and C by the heads of a group: G groups equal H groups
  with B, C repeated per head, dB and dC then summed over each group's heads;
* PyTorch's autograd in float64 over a direct sequential implementation
  (an independent library routine, a cross-check only).

The layer is the state-space recurrence of "Training Transformers and Hybrid
models on AMD Instinct MI300X Accelerators", section "Mamba-2" (the Mamba-2
selective scan with one decay per head); the pages print no worked example,
so every pin is mathematical.
"""

from __future__ import annotations

import numpy as np

from oracle import ssd

NAMES = ("x", "dt", "A", "B", "C", "D")


def make_case(rng, Bt=2, T=7, H=4, G=2, N=3, P=2, a_lo=0.3, a_hi=1.5):
    x = rng.standard_normal((Bt, T, H, P))
    dt = rng.uniform(0.05, 0.8, (Bt, T, H))
    A = -rng.uniform(a_lo, a_hi, H)
    B = rng.standard_normal((Bt, T, G, N))
    C = rng.standard_normal((Bt, T, G, N))
    D = rng.standard_normal(H)
    dy = rng.standard_normal((Bt, T, H, P))
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=D), dy


def _close(a, b, rtol, atol=0.0, what=""):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, "%s: shape %s vs %s" % (what, a.shape, b.shape)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    ref = max(float(np.max(np.abs(b))) if b.size else 0.0, 1e-300)
    assert np.all(np.isfinite(a)), what
    assert err <= rtol * ref + atol, "%s: max|err| %.3e > %.1e * %.3e + %.1e" % (
        what, err, rtol, ref, atol)


def _fb(lib, case, dy):
    return ssd.ssd_forward_backward(*(case[n] for n in NAMES), dy, lib=lib)


def dual_form(case, dy):
    """y and the gradients from the dual (quadratic) form, in numpy."""
    x, dt, A, B, C, D = (case[n] for n in NAMES)
    Bt, T, H, P = x.shape
    G = B.shape[2]
    hpg = H // G
    out = {k: np.zeros_like(case[k]) for k in ("x", "dt", "A", "B", "C", "D")}
    y = np.zeros_like(x)
    tri = np.tril(np.ones((T, T), bool))
    for b in range(Bt):
        for h in range(H):
            g = h // hpg
            cs = np.cumsum(dt[b, :, h])
            seg = cs[:, None] - cs[None, :]                      # cs_t - cs_s
            Lm = np.where(tri, np.exp(A[h] * np.where(tri, seg, 0.0)), 0.0)
            CB = C[b, :, g] @ B[b, :, g].T                       # [t, s]
            M = CB * Lm * dt[b, :, h][None, :]                   # y = M x + D x
            xs, dys = x[b, :, h], dy[b, :, h]
            y[b, :, h] = M @ xs + D[h] * xs
            YX = dys @ xs.T                                      # dy_t . x_s
            Gm = YX * M                                          # per-pair loss terms
            out["x"][b, :, h] = M.T @ dys + D[h] * dys
            W = YX * Lm * dt[b, :, h][None, :]
            out["C"][b, :, g] += W @ B[b, :, g]
            out["B"][b, :, g] += W.T @ C[b, :, g]
            out["D"][h] += np.sum(dys * xs)
            out["A"][h] += np.sum(Gm * np.where(tri, seg, 0.0))
            # dt_r: the explicit factor dt_s (s = r), and the decay: every pair
            # s < r <= t carries A * G_ts
            direct = np.sum(YX * CB * Lm, axis=0)                # over t, for s = r
            decay = np.zeros(T)
            for r in range(T):
                decay[r] = A[h] * np.sum(Gm[r:, :r])
            out["dt"][b, :, h] = direct + decay
    return y, out


def pin_finite_differences(lib):
    rng = np.random.default_rng(101)
    case, dy = make_case(rng, Bt=1, T=5, H=2, G=1, N=2, P=2)
    grads = _fb(lib, case, dy)

    def loss(c):
        return float(np.sum(dy * ssd.ssd_forward(*(c[n] for n in NAMES), lib=lib)))
    for name in NAMES:
        base = case[name]
        num = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            h = 1e-6 * max(1.0, abs(base[idx]))
            plus = {k: v.copy() for k, v in case.items()}
            minus = {k: v.copy() for k, v in case.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            num[idx] = (loss(plus) - loss(minus)) / (2 * h)
        _close(grads["d" + name], num, 1e-6, 1e-8, "finite differences d%s" % name)


def pin_dual_form(lib):
    rng = np.random.default_rng(102)
    for kw in (dict(), dict(Bt=1, T=12, H=3, G=1, N=4, P=3), dict(H=2, G=2, T=9)):
        case, dy = make_case(rng, **kw)
        o = _fb(lib, case, dy)
        y, g = dual_form(case, dy)
        _close(o["y"], y, 1e-12, what="dual y")
        _close(ssd.ssd_forward(*(case[n] for n in NAMES), lib=lib), y, 1e-12,
               what="dual y (forward only)")
        for name in NAMES:
            _close(o["d" + name], g[name], 1e-11, 1e-13, "dual d%s %s" % (name, kw))


def pin_closed_forms(lib):
    rng = np.random.default_rng(103)
    # one step: y = dt (C . B) x + D x and its gradients
    case, dy = make_case(rng, T=1)
    o = _fb(lib, case, dy)
    x, dt, A, B, C, D = (case[n] for n in NAMES)
    hpg = x.shape[2] // B.shape[2]
    Bh = np.repeat(B, hpg, axis=2)
    Ch = np.repeat(C, hpg, axis=2)
    cb = np.sum(Bh * Ch, axis=-1)                                  # [Bt, 1, H]
    _close(o["y"], (dt * cb)[..., None] * x + D[None, None, :, None] * x, 1e-13, what="T=1 y")
    _close(o["dx"], (dt * cb)[..., None] * dy + D[None, None, :, None] * dy, 1e-13,
           what="T=1 dx")
    _close(o["ddt"], cb * np.sum(dy * x, -1), 1e-13, what="T=1 ddt")
    _close(o["dA"], np.zeros_like(A), 0, 0, "T=1 dA")
    # no decay (A = 0): h_t = sum_{s <= t} dt_s B_s x_s^T
    case, dy = make_case(rng, T=6)
    case["A"] = np.zeros_like(case["A"])
    o = _fb(lib, case, dy)
    x, dt, B, C, D = case["x"], case["dt"], case["B"], case["C"], case["D"]
    hpg = x.shape[2] // B.shape[2]
    y = np.zeros_like(x)
    for b in range(x.shape[0]):
        for h in range(x.shape[2]):
            g = h // hpg
            state = np.zeros((B.shape[3], x.shape[3]))
            for t in range(x.shape[1]):
                state = state + dt[b, t, h] * np.outer(B[b, t, g], x[b, t, h])
                y[b, t, h] = state.T @ C[b, t, g] + D[h] * x[b, t, h]
    _close(o["y"], y, 1e-12, what="A=0 y")
    # a decay that underflows to zero: no memory
    case, dy = make_case(rng, T=6)
    case["A"] = np.full_like(case["A"], -1e5)
    o = _fb(lib, case, dy)
    x, dt, B, C, D = case["x"], case["dt"], case["B"], case["C"], case["D"]
    Bh = np.repeat(B, hpg, axis=2)
    Ch = np.repeat(C, hpg, axis=2)
    cb = np.sum(Bh * Ch, axis=-1)
    _close(o["y"], (dt * cb)[..., None] * x + D[None, None, :, None] * x, 1e-13,
           what="no memory y")
    _close(o["dA"], np.zeros_like(case["A"]), 0, 0, "no memory dA")


def pin_groups_share_b_and_c(lib):
    rng = np.random.default_rng(104)
    case, dy = make_case(rng, Bt=2, T=6, H=6, G=2, N=3, P=2)
    o = _fb(lib, case, dy)
    hpg = 3
    per_head = dict(case)
    per_head["B"] = np.repeat(case["B"], hpg, axis=2)
    per_head["C"] = np.repeat(case["C"], hpg, axis=2)
    o2 = _fb(lib, per_head, dy)
    for name in ("y", "dx", "ddt", "dA", "dD"):
        _close(o[name], o2[name], 1e-13, what="groups " + name)
    for name in ("dB", "dC"):
        summed = o2[name].reshape(2, 6, 2, hpg, 3).sum(axis=3)
        _close(o[name], summed, 1e-13, what="groups " + name)


def pin_torch_autograd(lib):
    try:
        import torch
    except ImportError:
        return
    rng = np.random.default_rng(105)
    case, dy = make_case(rng, Bt=2, T=8, H=4, G=2, N=3, P=2)
    o = _fb(lib, case, dy)
    t = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in case.items()}
    x, dt, A, B, C, D = (t[n] for n in NAMES)
    Bt, T, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    ys = []
    for h in range(H):
        g = h // hpg
        state = torch.zeros((Bt, N, P), dtype=torch.float64)
        yh = []
        for s in range(T):
            a = torch.exp(dt[:, s, h] * A[h])[:, None, None]
            state = a * state + dt[:, s, h][:, None, None] * B[:, s, g, :, None] * x[:, s, h, None, :]
            yh.append(torch.einsum("bnp,bn->bp", state, C[:, s, g]) + D[h] * x[:, s, h])
        ys.append(torch.stack(yh, 1))
    y = torch.stack(ys, 2)
    (y * torch.tensor(dy)).sum().backward()
    _close(o["y"], y.detach().numpy(), 1e-12, what="torch y")
    for name in NAMES:
        _close(o["d" + name], t[name].grad.numpy(), 1e-11, 1e-13, "torch d" + name)


ALL_PINS = [pin_finite_differences, pin_dual_form, pin_closed_forms, pin_groups_share_b_and_c,
            pin_torch_autograd]
