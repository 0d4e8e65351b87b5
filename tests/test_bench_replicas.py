"""The multi-GPU path of the benchmark on the CPU: N independent replicas
(the decode shards by sequence with no exchange), timed by the slowest rank.
Runs world_size-2 process groups over gloo on 127.0.0.1; the GPU kernels are
not involved, only the host logic that turns per-rank times into the job's
figure, and the reference arm's rank handling under torchrun."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [0.120, 0.135][rank]                 # rank 1 is the slow replica
        slowest = bench.max_over_ranks(mine, torch.device("cpu"), world)
        dist.barrier()
        out[rank] = (slowest, bench.replica_gbs(717.18e6 * 64, slowest * 64, world))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_summed_bytes():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    slowest, gbs = out[0]
    assert slowest == pytest.approx(0.135)
    assert gbs == pytest.approx(2 * 717.18e6 / 0.135 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, torch.device("cpu"), 1) == 1.5
    assert bench.replica_gbs(1e9, 1.0, 1) == pytest.approx(1.0)


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line_carries_the_contract_keys():
    """One GPU-less run of the reference arm (the oracle on the host cores):
    one JSON line with the bench contract's keys, its e2e equal to its own
    value with no host-device bytes, and a cpu_baseline describing the run."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_other_workloads_report_a_failure_instead_of_ending_the_line(monkeypatch):
    """The default line measures the INT8 and verification workloads after the
    headline; one that raises is recorded by its error and the rest still run."""
    sys.path.insert(0, ROOT)
    import bench
    seen = []

    def fake_measure(name, pa, W, torch_mod, dev, reps, warmup, partition=0, flush=None):
        seen.append(name)
        if name == bench.OTHER_WORKLOADS[1]:
            raise RuntimeError("synthetic failure")
        return {"workload": name, "attention_us": 1.0}

    monkeypatch.setattr(bench, "measure_workload", fake_measure)
    monkeypatch.setattr(bench, "l2_flusher", lambda torch_mod, dev: None)
    res = bench.measure_other_workloads(None, None, torch, torch.device("cpu"))
    assert seen == bench.OTHER_WORKLOADS
    assert "synthetic failure" in res[bench.OTHER_WORKLOADS[1]]["error"]
    for name in bench.OTHER_WORKLOADS[:1] + bench.OTHER_WORKLOADS[2:]:
        assert res[name]["attention_us"] == 1.0
    from paged_kv_decode_27_gb300 import workloads as W
    for name in bench.OTHER_WORKLOADS:
        assert name in W.WORKLOADS and name in bench.N_LAYERS
