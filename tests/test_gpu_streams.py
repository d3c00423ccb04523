"""Stream behaviour of the GPU path: the kernels are launched with
programmatic dependent launch (each may start its set-up while the previous
kernel in the stream finishes, and waits for it before reading memory).

- Back-to-back calls on one stream, where each call's inputs are the previous
  call's outputs, must see the finished outputs.
- A CUDA graph captured from attn_fwd + attn_bwd (the programmatic launches
  become graph edges) must replay to the same bits as the eager calls.
- Two independent problems on two streams must not interfere.
"""

import pytest
import torch

from attention_backward_pass_attn_gb300 import binding as ab
from attention_backward_pass_attn_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_backward_pass_attn_gb300 import build as abuild

    abuild.build()
    ab.load_library()


def device_inputs(name, seed_shift=0.0):
    w = WORKLOADS[name]
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    if seed_shift:
        q = (q.float() + seed_shift).to(torch.bfloat16)
    return w, q, k, v, do


def test_chained_calls_see_finished_outputs():
    """O of one forward is the Q of the next, five times over, with no host
    synchronisation between the calls; the same chain with a device
    synchronisation after every call gives the same bits."""
    w, q, k, v, do = device_inputs("b2h16n2048d64_causal")

    def chain(sync):
        x = q
        outs = []
        for _ in range(5):
            o, lse = ab.attn_fwd(x, k, v, w.causal, w.scale)
            if sync:
                torch.cuda.synchronize()
            dq, dk, dv = ab.attn_bwd(x, k, v, o, do, lse, w.causal, w.scale)
            if sync:
                torch.cuda.synchronize()
            outs.append((o, dk, dv))
            x = o  # the next call reads what this one wrote
        torch.cuda.synchronize()
        return outs

    eager = chain(False)
    synced = chain(True)
    for (o1, dk1, dv1), (o2, dk2, dv2) in zip(eager, synced):
        assert torch.equal(o1, o2) and torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert ab.attn_last_device_error() == ab.ATTN_OK


def test_graph_replay_matches_eager():
    w, q, k, v, do = device_inputs("b1h2n128d64")
    ws = ab.alloc_workspace(w.B, w.H, w.N, w.d, q.device)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=q.device)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    stream = torch.cuda.Stream()

    def step():
        ab.attn_fwd(q, k, v, w.causal, w.scale, out=o, lse=lse, stream=stream)
        ab.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, dq=dq, dk=dk, dv=dv, workspace=ws,
                    stream=stream)

    with torch.cuda.stream(stream):
        step()  # eager, also resolves the library's one-time look-ups before capture
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dk, dv, dq)]
    for t in (o, dq, dk, dv):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    got = (o, lse, dk, dv, dq)
    for a, b in zip(got[:4], ref[:4]):
        assert torch.equal(a, b)  # forward, dK, dV: one CTA each, bitwise repeatable
    # dQ partials are added with fp32 reductions across CTAs: order may differ
    err = float((got[4].double() - ref[4].double()).abs().max() / ref[4].double().abs().max())
    assert err <= 2e-3
    assert ab.attn_last_device_error(stream) == ab.ATTN_OK


def test_two_streams_do_not_interfere():
    w, q1, k, v, do = device_inputs("b2h16n2048d64_causal")
    _, q2, _, _, _ = device_inputs("b2h16n2048d64_causal", seed_shift=0.25)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    refs = []
    for q in (q1, q2):
        o, lse = ab.attn_fwd(q, k, v, w.causal, w.scale)
        refs.append((o,) + ab.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale))
    torch.cuda.synchronize()
    outs = []
    for q, s in ((q1, s1), (q2, s2)):
        with torch.cuda.stream(s):
            o, lse = ab.attn_fwd(q, k, v, w.causal, w.scale, stream=s)
            outs.append((o,) + ab.attn_bwd(q, k, v, o, do, lse, w.causal, w.scale, stream=s))
    torch.cuda.synchronize()
    for (o, dq, dk, dv), (ro, rdq, rdk, rdv) in zip(outs, refs):
        assert torch.equal(o, ro) and torch.equal(dk, rdk) and torch.equal(dv, rdv)
        err = float((dq.double() - rdq.double()).abs().max() / rdq.double().abs().max())
        assert err <= 2e-3
    assert ab.attn_last_device_error() == ab.ATTN_OK
