"""Seeded synthetic inputs and the named attention workloads.

This module holds no attention arithmetic: it only draws random numbers and
describes shapes.  Both the CUDA path and the fp64 oracle are fed from here,
so they always see the same bf16 values.

Recipe (one rule for every workload): a CPU ``torch.Generator`` seeded with
the workload's seed draws ``torch.randn`` float32 tensors in the order Q, K,
V, dO, each of shape [B, H, N, d]; the workload's scale factors are applied in
float32; each tensor is then rounded once, to nearest even, to bfloat16.
Standard-normal inputs follow the benchmarking method of "Training - CUDA
Moat Still Alive" (section on the GEMM benchmark: inputs drawn from a normal
distribution with mean 0 and variance 1).
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    q_scale: float = 1.0   # Q is multiplied by this before the bf16 cast
    do_scale: float = 1.0  # dO is multiplied by this before the bf16 cast
    window: int = 0        # causal sliding window (0 = none)
    doc_lengths: tuple = ()  # causal documents packed in order (empty = one document)

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d)."""
        return 1.0 / math.sqrt(self.d)

    @property
    def heads(self) -> int:
        return self.B * self.H

    def pairs(self) -> float:
        """Visible (query, key) pairs per head: N^2, N^2/2 under the causal
        mask, N*W - W^2/2 (the area of the band) under a window W < N, and
        the sum of n^2/2 over packed documents of lengths n."""
        N, W = float(self.N), float(self.window)
        if self.causal and self.doc_lengths:
            return sum(float(n) * n / 2 for n in self.doc_lengths)
        if self.causal and 0 < W < N:
            return N * W - W * W / 2
        return N * N / 2 if self.causal else N * N

    def fwd_flops(self) -> float:
        """4*d FLOPs per visible pair: 4*B*H*N^2*d, halved under the causal mask."""
        return 4.0 * self.B * self.H * self.d * self.pairs()

    def bwd_flops(self) -> float:
        """10*d FLOPs per visible pair (five contractions): 10*B*H*N^2*d, halved
        under the causal mask."""
        return 10.0 * self.B * self.H * self.d * self.pairs()

    def describe(self) -> str:
        return ("B=%d H=%d N=%d d=%d %s%s q_scale=%g do_scale=%g seed=%d"
                % (self.B, self.H, self.N, self.d,
                   "causal" if self.causal else "non-causal",
                   " window=%d" % self.window if self.window else "",
                   self.q_scale, self.do_scale, self.seed))

    def with_shape(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads the parity tests and the benchmark use, named by shape.
WORKLOADS = {
    "b1h2n128d64": Workload("b1h2n128d64", 1, 2, 128, 64, False, seed=0),
    "b2h16n2048d64_causal": Workload("b2h16n2048d64_causal", 2, 16, 2048, 64, True, seed=1),
    "b1h32n4096d128_causal": Workload("b1h32n4096d128_causal", 1, 32, 4096, 128, True,
                                      seed=2, do_scale=0.1),
    "b4h16n8192d128": Workload("b4h16n8192d128", 4, 16, 8192, 128, False, seed=3,
                               q_scale=2.0),
    "b1h16n16384d128_causal": Workload("b1h16n16384d128_causal", 1, 16, 16384, 128, True,
                                       seed=4),
}
WORKLOAD_ORDER = list(WORKLOADS)

def _packed_lengths(N: int, lo: int, hi: int, seed: int) -> tuple:
    """Document lengths drawn uniformly from [lo, hi] until N positions are
    filled (the last one cut to fit): a seeded packing of variable-length
    sequences."""
    g = torch.Generator().manual_seed(seed)
    out = []
    while sum(out) < N:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(min(n, N - sum(out)))
    return tuple(out)


# Mask variants measured beside the workloads above: sliding-window attention
# at the Mistral 7B window (4096 keys), and packed documents of 512 to 4096
# positions.
EXTRA_WORKLOADS = {
    "b1h16n16384d128_w4096": Workload("b1h16n16384d128_w4096", 1, 16, 16384, 128, True,
                                      seed=5, window=4096),
    "b1h16n16384d128_docs": Workload("b1h16n16384d128_docs", 1, 16, 16384, 128, True, seed=6,
                                     doc_lengths=_packed_lengths(16384, 512, 4096, seed=6)),
}


def make_doc_map(w: Workload) -> torch.Tensor | None:
    """The document map of a workload, int32 [B, N] (the first position of
    each position's document; the same packing for every batch element), or
    None for one document."""
    if not w.doc_lengths:
        return None
    starts = []
    pos = 0
    for n in w.doc_lengths:
        starts.extend([pos] * n)
        pos += n
    return torch.tensor(starts, dtype=torch.int32).repeat(w.B, 1)


def make_inputs(w: Workload, dtype=torch.bfloat16):
    """Return (q, k, v, do) CPU tensors of shape [B, H, N, d] in ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    shape = (w.B, w.H, w.N, w.d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    if w.q_scale != 1.0:
        q.mul_(w.q_scale)
    if w.do_scale != 1.0:
        do.mul_(w.do_scale)
    return tuple(t.to(dtype) for t in (q, k, v, do))


def make_tensor(shape, seed: int, dtype=torch.bfloat16, std: float = 1.0):
    """One seeded N(0, std^2) tensor, for edge-case tests."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def quantize_e4m3(t: torch.Tensor):
    """An 8-bit (OCP FP8 E4M3) copy of a tensor with one per-tensor descale
    factor: descale = max|t| / 448 (448 is e4m3's largest finite value) as an
    fp32 number, bytes = round-to-nearest-even(t / descale), so that
    bytes x descale stands for t.  Returns (float8_e4m3fn tensor, descale).
    Input preparation for the fp8 entry point: the tensors the caller hands
    it, not attention arithmetic."""
    x = t.to(torch.float32)
    amax = float(x.abs().max()) if x.numel() else 0.0
    descale = float(torch.tensor(amax / 448.0 if amax > 0 else 1.0, dtype=torch.float32))
    return (x / descale).to(torch.float8_e4m3fn), descale


def make_inputs_fp8(w: Workload):
    """The workload's seeded inputs (make_inputs, bf16) quantised to e4m3 with
    a per-tensor descale each: ((q8, qd), (k8, kd), (v8, vd), do)."""
    q, k, v, do = make_inputs(w)
    return quantize_e4m3(q), quantize_e4m3(k), quantize_e4m3(v), do


# --------------------------------------------------------------------------
# The Mamba-2 state-space layer (the hybrid model's second hot kernel).
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class SsdWorkload:
    """Shapes of one Mamba-2 layer: Bt sequences of T steps, H heads of P
    channels, G groups of B/C with a state of N per channel."""
    name: str
    Bt: int
    T: int
    H: int
    G: int
    N: int
    P: int
    seed: int

    @property
    def tokens(self) -> int:
        return self.Bt * self.T

    def recurrence_flops(self) -> float:
        """FLOPs of the backward written as the recurrence and its adjoint:
        per (b, t, h) the state update and the suffix update (2 NP each),
        dx, dB, dC (2 NP each), ddt and dA (5 NP), the recomputed forward
        state (2 NP): 17 N P."""
        return 17.0 * self.Bt * self.T * self.H * self.N * self.P


SSD_WORKLOADS = {
    # d_model 2048 with expansion 2 (4096 channels = 64 heads of 64), state
    # 128, one group: at the three sequence lengths the pages measure.
    "ssd_b2t2048h64n128": SsdWorkload("ssd_b2t2048h64n128", 2, 2048, 64, 1, 128, 64, seed=21),
    "ssd_b2t4096h64n128": SsdWorkload("ssd_b2t4096h64n128", 2, 4096, 64, 1, 128, 64, seed=22),
    "ssd_b1t8192h64n128": SsdWorkload("ssd_b1t8192h64n128", 1, 8192, 64, 1, 128, 64, seed=23),
}


def make_ssd_inputs(w: SsdWorkload):
    """(x, dt, A, B, C, D, dy) as CPU tensors: x, B, C, dy standard normal,
    rounded once to bf16; dt log-uniform in [1e-3, 1e-1] and A uniform in
    [-16, -1] (Mamba-2's initialisation ranges), D uniform in [0.5, 1.5], all
    fp32."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(w.seed))
    x = torch.randn((w.Bt, w.T, w.H, w.P), generator=g, dtype=torch.float32)
    B = torch.randn((w.Bt, w.T, w.G, w.N), generator=g, dtype=torch.float32)
    C = torch.randn((w.Bt, w.T, w.G, w.N), generator=g, dtype=torch.float32)
    dy = torch.randn((w.Bt, w.T, w.H, w.P), generator=g, dtype=torch.float32)
    u = torch.rand((w.Bt, w.T, w.H), generator=g, dtype=torch.float32)
    dt = torch.exp(math.log(1e-3) + u * (math.log(1e-1) - math.log(1e-3)))
    A = -(1.0 + 15.0 * torch.rand((w.H,), generator=g, dtype=torch.float32))
    D = 0.5 + torch.rand((w.H,), generator=g, dtype=torch.float32)
    bf = torch.bfloat16
    return x.to(bf), dt, A, B.to(bf), C.to(bf), D, dy.to(bf)
