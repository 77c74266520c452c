"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The layer shards over (batch, head) and over whole layer calls with no
exchange in the data path, so a run on N GPUs is N independent replicas
(weak scaling): the only cross-rank steps are the barrier around the timed
region and the max over ranks of the measured time. These run here as two
gloo processes on 127.0.0.1.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r measured (r + 1) ms: the job's time is the slowest rank's
        ms = bench.max_over_ranks(float(rank + 1), dist, torch.device("cpu"))
        rate = bench.job_throughput(1000.0, world, ms)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_rate_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, rate in res:
        assert ms == 2.0
        assert rate == pytest.approx(1000.0 * 2 / 2e-3)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    import lact_inputs as li
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus = 1, 0, 2
    assert bench.run_reference(Args(), li.WORKLOADS[1]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_has_the_contract_keys():
    # rank 0 of a one-process run prints one JSON line in the bench's unit
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                         env={k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "tiny-causal-f32-gd"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "sample" in cb
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_context_parallel_bench_rejects_the_causal_order():
    # the context-parallel mode spreads one set-order update chunk over the
    # ranks; a causal layer (a chain of chunks) is refused before any GPU work
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--context-parallel", "--workload", "2"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "set order" in (r.stderr + r.stdout)
