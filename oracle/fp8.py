"""Decoding of 8-bit floating-point inputs for the fp64 oracle.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): only the test suite,
the smoke check and the benchmark's CPU-baseline leg may import it.  It shares
no code with the CUDA path.

The fp8 forward of the CUDA library takes OCP FP8 E4M3 bytes with one fp32
descale factor per tensor.  What it computes is exact attention of the values
those bytes stand for, so the oracle decodes them to float64 (exactly: every
E4M3 value times an fp32 factor has at most 28 significant bits) and runs the
same exact-attention oracle on them.

E4M3 (the "FN" variant, no infinities), from the format's definition: bit 7
sign, bits 6-3 biased exponent e (bias 7), bits 2-0 mantissa m.
  e = 0:            (-1)^s * m/8 * 2^(1-7)       (zero and subnormals)
  e = 15, m = 7:    NaN
  otherwise:        (-1)^s * (1 + m/8) * 2^(e-7)  (largest finite: 448)
"""

from __future__ import annotations

import numpy as np


def e4m3_to_f64(codes) -> np.ndarray:
    """float64 values of E4M3 byte codes (any integer array of 0..255)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    sub = m / 8.0 * 2.0 ** (1 - 7)
    norm = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    out = sign * np.where(e == 0, sub, norm)
    return np.where((e == 15) & (m == 7), np.nan, out)


def dequantize(t8, descale: float) -> np.ndarray:
    """The values a tensor of E4M3 bytes with a per-tensor descale factor
    stands for, in float64: code value x descale.  Accepts a torch tensor
    (float8_e4m3fn or uint8) or a numpy array of codes."""
    if hasattr(t8, "detach"):
        import torch  # local: the decoder itself does not need torch

        t8 = t8.detach().to("cpu")
        if t8.dtype != torch.uint8:
            t8 = t8.view(torch.uint8)
        t8 = t8.numpy()
    return e4m3_to_f64(t8) * float(descale)
