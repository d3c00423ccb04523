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

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d)."""
        return 1.0 / math.sqrt(self.d)

    @property
    def heads(self) -> int:
        return self.B * self.H

    def pairs(self) -> float:
        """Visible (query, key) pairs per head: N^2, N^2/2 under the causal
        mask, and N*W - W^2/2 (the area of the band) under a window W < N."""
        N, W = float(self.N), float(self.window)
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

# Sliding-window attention at the Mistral 7B window (4096 keys), measured
# beside the workloads above.
EXTRA_WORKLOADS = {
    "b1h16n16384d128_w4096": Workload("b1h16n16384d128_w4096", 1, 16, 16384, 128, True,
                                      seed=5, window=4096),
}


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
