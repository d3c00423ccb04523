"""Host-side logic of bench.py, on the CPU: the multi-rank aggregation (two
gloo ranks), clock-record parsing, the ncu-traffic staleness check, and the
reference arm on the smallest workload."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _agg_worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r took 10*(r+1) ms for r+1 units of work
    t, f = bench.aggregate(10.0 * (rank + 1), float(rank + 1))
    q.put((rank, t, f))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29400 + os.getpid() % 500
    procs = [ctx.Process(target=_agg_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    # slowest rank's time, all ranks' work, seen identically by both ranks
    assert got == [(0, 20.0, 3.0), (1, 20.0, 3.0)]


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(5.0, 7.0) == (5.0, 7.0)


def test_clock_parsing():
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop()["sm_mhz"] is None

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = FakeProc()
    s.lines = ["0, 1900, 2070, 900.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "0, 1950, 2070, 1000.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1800, 2070, 1100.0, 0x0, Active, Not Active, Not Active, Not Active",
               "garbage"]
    r = s.stop()
    assert r["sm_mhz"] == 1900 and r["sm_max_mhz"] == 2070 and r["samples"] == 3
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_stored_traffic_requires_current_sources(tmp_path, monkeypatch):
    """A stored ncu traffic figure is reported only while the CUDA sources
    still hash to the value recorded with it."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel=None: "current")
    (prof / "ncu_traffic.json").write_text(json.dumps({
        "k@w": {"source_hash": "stale", "dram_bytes_per_launch": 123},
        "k2@w": {"source_hash": "current", "dram_bytes_per_launch": 456}}))
    assert bench.stored_traffic("k", "w") is None
    assert bench.stored_traffic("k2", "w") == 456
    assert bench.stored_traffic("missing", "w") is None


def test_kernel_hash_covers_its_sources(tmp_path, monkeypatch):
    """A kernel's hash changes with its own sources and ignores comments and
    the files it is not built from."""
    csrc = tmp_path / "attention_backward_pass_attn_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ["a.cu", "p.cuh"]})
    (csrc / "a.cu").write_text("int a = 1;  // note\n")
    (csrc / "p.cuh").write_text("#pragma once\n")
    (csrc / "other.cu").write_text("int b = 2;\n")
    h0 = bench.kernel_source_hash("k")
    (csrc / "a.cu").write_text("int a = 1;  // another note\n")
    (csrc / "other.cu").write_text("int b = 3;\n")
    assert bench.kernel_source_hash("k") == h0
    (csrc / "a.cu").write_text("int a = 2;\n")
    assert bench.kernel_source_hash("k") != h0


def test_committed_ncu_entries_match_their_sources():
    """Every committed ncu entry names a kernel whose CUDA sources are known and
    still hash to the value recorded with it: a kernel change needs a new
    capture (or the entry's removal) before its counters are reported."""
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    assert table
    for key, ent in table.items():
        kernel, _, workload = key.partition("@")
        assert workload, key
        assert kernel in bench.KERNEL_SOURCES, key
        assert ent["source_hash"] == bench.kernel_source_hash(kernel), key
        assert ent["dram_bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"], key
        assert "--clock-control none" in ent["command"], key
        assert bench.stored_ncu(kernel, workload) is ent or bench.stored_ncu(kernel, workload) == ent


def test_reference_arm_runs_on_cpu():
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "b1h2n128d64", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "b1h2n128d64", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, env=env)
    assert p.returncode == 0 and p.stdout.strip() == ""


def _visible_pairs(N, causal, window=0, lengths=()):
    """Brute-force count of the (query, key) pairs the mask lets through."""
    doc = []
    for n in lengths:
        doc += [len(doc)] * n
    count = 0
    for i in range(N):
        for j in range(N):
            if causal and j > i:
                continue
            if window and i - j >= window:
                continue
            if lengths and doc[j] < doc[i]:
                continue
            count += 1
    return count


@pytest.mark.parametrize("N,causal,window,lengths", [
    (37, False, 0, ()), (37, True, 0, ()), (64, True, 9, ()), (64, True, 64, ()),
    (50, True, 0, (20, 1, 29)), (128, True, 0, (128,))])
def test_flop_pairs_follow_the_mask(N, causal, window, lengths):
    """The FLOP accounting counts the area of the visible region: the brute-force
    pair count minus half of its diagonal band (N^2/2 under the causal mask, the
    usual convention), so both arms are measured against the same work."""
    from attention_backward_pass_attn_gb300.inputs import Workload

    w = Workload("t", 1, 1, N, 64, causal, seed=0, window=window, doc_lengths=lengths)
    exact = _visible_pairs(N, causal, window, lengths)
    if not causal:
        assert w.pairs() == exact
    elif 0 < window < N:
        assert w.pairs() == exact - window / 2
    else:
        assert w.pairs() == exact - N / 2
    assert w.bwd_flops() == 10 * 64 * w.pairs() and w.fwd_flops() == 4 * 64 * w.pairs()
