"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a host framework whose allocator owns all device memory and hands a
plug-in only its tensors, or a latency-bound loop that cannot afford
cudaMalloc's implicit synchronisation).  It takes no workspace and uses the
library's own fixed 32 MiB device scratch instead.

Called through the C ABI and compared with attn_bwd (which takes a caller
workspace) on the same inputs, on two calls in a row with different inputs,
so that anything the first call leaves in the shared scratch would show up
in the second.  This file is collected last on purpose.
"""

import ctypes

import numpy as np
import pytest
import torch

from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

TOL = 1e-2  # same bound as the parity tests: max|a - b| / max|b|


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_backward_pass_attn_gb300 import build as abuild

    abuild.build()
    return ab.load_library()


def rel(a, b):
    a = a.to(torch.float64)
    b = b.to(torch.float64)
    return float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))


def noalloc_bwd(lib, q, k, v, o, do, lse, causal, scale):
    B, H, N, d = q.shape
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, int(causal), float(scale), stream)
    assert st == ab.ATTN_OK, lib.attn_status_string(st)
    return dq, dk, dv


def test_noalloc_matches_workspace_backward_twice(lib):
    dev = torch.device("cuda", 0)
    for name, seed in (("b2h16n2048d64_causal", 1), ("b2h16n2048d64_causal", 77),
                       ("b1h2n128d64", 0)):
        w = WORKLOADS[name].with_shape(seed=seed)
        q, k, v, do = (t.to(dev) for t in make_inputs(w))
        o, lse = ab.attn_fwd(q, k, v, w.causal, w.scale)
        ref = ab.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale)
        got = noalloc_bwd(lib, q, k, v, o, do, lse, w.causal, w.scale)
        torch.cuda.synchronize()
        assert lib.attn_last_device_error(None) == ab.ATTN_OK
        for g, r, n in zip(got, ref, ("dQ", "dK", "dV")):
            e = rel(g, r)
            assert np.isfinite(e) and e <= TOL, "%s seed %d %s: %.3e" % (name, seed, n, e)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    w = WORKLOADS["b1h32n4096d128_causal"]  # needs about 68 MB of workspace
    assert lib.attn_bwd_workspace_size(w.B, w.H, w.N, w.d) > (32 << 20)
    dev = torch.device("cuda", 0)
    t = torch.empty((1, 1, 1, 8), dtype=torch.bfloat16, device=dev)  # never touched
    p = t.data_ptr()
    st = lib.attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, w.B, w.H, w.N, w.d, 1, w.scale, None)
    assert st == ab.ATTN_ERR_TOO_LARGE
    assert b"32 MiB" in lib.attn_status_string(st)
