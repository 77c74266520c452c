"""Benchmark of the LaCT fast-weight chunk step on B300 (liblact, sm_103a).

One step = one whole layer call (lact_sequence) over one batch of synthetic
input: for the million-token set workload, the chunk gradient over 1,048,576
update tokens per head (8 heads, d=128, dh=512), one Muon step (5-step
Newton-Schulz) with row renorm, then the readout of 65,536 query tokens.

Prints ONE JSON line (rank 0). `value` is update+apply tokens/s over all
ranks with inputs resident in HBM; `e2e` is the same metric through the
public API with host (pinned) buffers, host<->device copies inside the timed
region. Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (no collective in the data path: weak scaling).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
                  [--impl lact|reference]

--impl reference times the fp64 CPU oracle (the only reference there is) on
a bounded sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import lact_inputs as li  # noqa: E402

METRIC = "TTT-layer tokens/sec (update+apply); tensor TFLOP/s vs B300 dense BF16 peak"
L2_BYTES = 126 * 1024 * 1024
UNIT = "tokens/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", type=int, default=5)
    p.add_argument("--impl", default="lact", choices=["lact", "reference"])
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--no-cpu-baseline", action="store_true")
    # time direct lact_sequence calls instead of a CUDA-graph replay of one
    p.add_argument("--no-graph", action="store_true")
    # one update chunk spread over the ranks by tokens (each rank's slice
    # gradient, one all-reduce of the gradients, the same update everywhere;
    # queries split likewise): strong scaling of one layer call. Set order only.
    p.add_argument("--context-parallel", action="store_true")
    # smaller token counts of the same layer (for profiler captures of a small case)
    p.add_argument("--update-tokens", type=int, default=None)
    p.add_argument("--query-tokens", type=int, default=None)
    return p.parse_args()


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float, pg, device) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's)."""
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job rate: every rank processes its own units (weak scaling)."""
    return units_per_rank * world / (ms / 1e3)


def flops(w: li.Workload) -> dict:
    """Algorithmic FLOP of one layer call (per the method, no recompute)."""
    BH, d, dh = w.B * w.H, w.d, w.dh
    chunks = -(-w.n_kv // w.chunk) if w.order == "causal" else 1
    if w.memory == "linear":
        # o = W q: 2 d^2 per query; dW = -(eta V)^T K: 2 d^2 per update token
        upd, app, nmat = 2 * d * d * w.n_kv * BH, 2 * d * d * w.n_q * BH, 1
    else:
        upd, app, nmat = 12 * d * dh * w.n_kv * BH, 6 * d * dh * w.n_q * BH, 3
    m, n = min(d, dh), max(d, dh)
    ns = (5 * (4 * m * m * n + 2 * m ** 3) * nmat * BH * chunks) if w.opt == "muon" else 0
    return {"update": upd, "apply": app, "ns": ns, "total": upd + app + ns}


def tokens_per_step(w: li.Workload) -> int:
    # causal tokens are both read and used for the update: count each once
    # (a layer token is processed by every head, so heads do not multiply it)
    per = w.n_kv if w.order == "causal" else w.n_kv + w.n_q
    return w.B * per


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one
# full-size launch of the fused gradient kernel on the million-token layer,
# scaled from an ncu capture of a reduced launch (131,072 tokens per head, 9
# token splits): reads (K, V, eta) grow with the tokens (x 8), writes (the
# split-K partial sums) with the splits (23 at full size). It describes the
# kernel source it was taken on, identified by its hash.
GRAD_TRAFFIC = {"workload": 5, "bytes": 560231168 * 8 + 46721536 * 23 // 9, "kernel_source": "k_tc_grad.cu",
                "sha256_prefix": "595c084a655bb093"}


def measured_traffic(w: li.Workload, reduced: bool):
    import hashlib
    if reduced or w.number != GRAD_TRAFFIC["workload"]:
        return None
    path = os.path.join(ROOT, "chunk_test_step_b300", "csrc", GRAD_TRAFFIC["kernel_source"])
    try:
        sha = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return GRAD_TRAFFIC["bytes"] if sha.startswith(GRAD_TRAFFIC["sha256_prefix"]) else None


FP64_TFLOPS = 1.25          # B300 dense fp64, nominal
BF16_MAC_PER_CLK_SM = 4096  # dense bf16 tensor-core MACs per clock per SM


def dense_bf16_tflops(sm_mhz: float, sms: int = 148) -> float:
    """Dense bf16 tensor rate at a given SM clock: SMs x 4,096 MACs x 2 FLOP."""
    return sms * BF16_MAC_PER_CLK_SM * 2 * sm_mhz * 1e6 / 1e12


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2032.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def pinned_inputs(w, inp):
    import torch

    def t(a):
        if a.dtype == np.uint16:
            x = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        else:
            x = torch.from_numpy(a)
        return x.pin_memory()
    return t(inp.q), t(inp.k), t(inp.v), t(inp.eta)


def blas_threads() -> int:
    """Threads numpy's BLAS uses (the oracle's only parallel part)."""
    try:
        from threadpoolctl import threadpool_info
        n = sum(x.get("num_threads", 0) for x in threadpool_info() if x.get("user_api") == "blas")
        if n:
            return n
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    # OpenBLAS default: one thread per available core, capped at its build limit (64)
    return min(len(os.sched_getaffinity(0)), 64)


def oracle_sample(w: li.Workload, n_kv: int) -> li.Workload:
    """One (b, h) of the workload with about n_kv update tokens (the workload's
    update:query ratio for set layers, whole chunks for causal layers)."""
    if w.order == "causal":
        n = max(w.chunk, min(w.n_kv, n_kv) // w.chunk * w.chunk)
        s = w.with_tokens(n, seed=w.seed + 7)
    else:
        n = max(1024, min(w.n_kv, n_kv) // 1024 * 1024)
        s = w.with_tokens(n, n_q=max(1, w.n_q * n // w.n_kv), seed=w.seed + 7)
    return dataclasses.replace(s, B=1, H=1)


def time_oracle(s: li.Workload) -> float:
    from oracle import lact_oracle as O
    inp = li.make_inputs(s)
    t0 = time.perf_counter()
    O.run_workload(s, inp, token_slice=65536)
    return time.perf_counter() - t0


def size_sample(w: li.Workload, seconds: float) -> li.Workload:
    """A sample of the workload sized for about `seconds` of oracle time:
    timed calibration runs from 16,384 update tokens, grown (at most 8x per
    run, since small runs carry a fixed cost) until one takes over half the
    target."""
    s = oracle_sample(w, 16384)
    while True:
        dt = max(time_oracle(s), 1e-3)
        if dt >= 0.5 * seconds or s.n_kv >= w.n_kv:
            break
        s = oracle_sample(w, int(s.n_kv * min(8.0, seconds / dt)))
    return oracle_sample(w, int(s.n_kv * seconds / dt))


def cpu_baseline(w: li.Workload, seconds: float = 15.0, sample: li.Workload | None = None):
    """The oracle, as it stands, on a bounded sample of the workload (one
    (b, h), sized for about `seconds` of CPU time)."""
    s1 = sample or size_sample(w, seconds)
    dt = time_oracle(s1)
    toks = tokens_per_step(s1)
    # A layer token is worked on by every one of the layer's H heads, and the
    # oracle takes one (b, h) after another: the layer's rate is the sample's
    # per-head rate over H (batch entries scale tokens and time alike).
    return {"value": toks / dt / w.H, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"1 (b,h) of the workload: {s1.n_kv} update + {s1.n_q if s1.order == 'set' else 0} "
                      f"query tokens, d={s1.d}, dh={s1.dh}, {s1.opt}, {s1.order}; fp64 numpy/OpenBLAS; "
                      f"{dt:.2f} s; value = sample tokens / (time x {w.H} heads), the oracle taking one "
                      f"(b, h) at a time",
            "seconds": dt}


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    # each step a sample sized so that the whole run takes about two minutes
    per_step = min(20.0, max(2.0, 120.0 / max(1, args.warmup + args.steps)))
    sample = size_sample(w, per_step)
    res = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(w, sample=sample)
        if i >= args.warmup:
            res.append(r)
    val = statistics.median(r["value"] for r in res)
    ms = statistics.median(r["seconds"] for r in res) * 1e3
    cb = dict(res[-1]); cb["value"] = val; cb.pop("seconds", None)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": cb["sample"]},
            "cpu_baseline": cb,
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_context_parallel(args, w):
    """One layer call of a set-order workload spread over the ranks by tokens.

    Rank r holds tokens token_range(n_kv, r, N) of the update chunk and
    token_range(n_q, r, N) of the queries (both [B, H, slice, d]); per step it
    computes its slice gradient, the ranks all-reduce the gradients (NCCL),
    every rank applies the same update, then reads its queries. The job's
    time is the slowest rank's; `value` is the whole layer's tokens over it
    (strong scaling: the work is one call whatever N is)."""
    import torch
    from chunk_test_step_b300 import lact as L
    from chunk_test_step_b300.context_parallel import ContextParallelUpdate, token_range
    if w.order != "set":
        raise SystemExit("--context-parallel serves the set order (one update chunk, then queries)")
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    inp = li.make_inputs(w)
    t0, t1 = token_range(w.n_kv, rank, world)
    q0, q1 = token_range(w.n_q, rank, world)
    hq, hk, hv, he = pinned_inputs(w, li.Inputs(np.ascontiguousarray(inp.q[:, :, q0:q1]),
                                                np.ascontiguousarray(inp.k[:, :, t0:t1]),
                                                np.ascontiguousarray(inp.v[:, :, t0:t1]),
                                                np.ascontiguousarray(inp.eta[:, :, t0:t1]), None, None, None))
    q, k, v, e = (x.to(dev) for x in (hq, hk, hv, he))
    n_loc, nq_loc = t1 - t0, q1 - q0
    W1, W2, W3 = (None if x is None else torch.from_numpy(x).to(dev) for x in (inp.W1, inp.W2, inp.W3))
    del inp
    cfg = L.make_config(w.B, w.H, w.d, w.dh, w.dtype, w.opt, max_chunk=max(1, n_loc), ns_steps=w.ns_steps,
                        ns_a=w.ns_a, ns_b=w.ns_b, ns_c=w.ns_c, muon_lr=w.muon_lr, momentum=w.momentum,
                        memory=w.memory)
    layer = L.LactLayer(cfg, W1, W2, W3, device=dev)
    cp = ContextParallelUpdate(layer, group=None if pg is None else pg.group.WORLD)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def step():
        cp.update(k, v, e, n_loc, stream)
        L.lact_chunk_apply(layer.handle, q, nq_loc, o, stream)

    def barrier():
        if pg:
            pg.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    def timed(run, n):
        barrier()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            run()
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        return a.elapsed_time(b)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    n0 = L.lact_launch_count()
    ms_step = max_over_ranks(timed(step, args.steps), pg, dev) / args.steps
    launches = L.lact_launch_count() - n0
    ck = clocks.stop()
    L.lact_set_profiling(layer.handle, True)
    timed(step, args.steps)
    prof = L.lact_get_profile(layer.handle)
    L.lact_set_profiling(layer.handle, False)

    def e2e_step():
        for d_, h_ in ((q, hq), (k, hk), (v, hv), (e, he)):
            d_.copy_(h_, non_blocking=True)
        step()
        ho.copy_(o, non_blocking=True)

    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    e2e_ms = max_over_ranks(timed(e2e_step, args.e2e_steps), pg, dev) / args.e2e_steps
    st = L.lact_sync_status(layer.handle)
    if st != L.LACT_OK:
        raise RuntimeError(f"device status after the timed region: {L.lact_status_str(st)}")

    pk, pk_src = peaks()
    grad = prof["grad"]
    grad_ms = grad["ms"] / max(1, grad["calls"])
    grad_flop = flops(w.with_tokens(n_loc, n_q=nq_loc))["update"]
    achieved = grad_flop / (grad_ms / 1e3) / 1e12
    tok = w.B * (w.n_kv + w.n_q)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, he))
    line = {"metric": METRIC, "value": tok / (ms_step / 1e3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d, "dh": w.dh,
                       "update_tokens_per_head": w.n_kv, "query_tokens_per_head": w.n_q,
                       "update_tokens_per_rank": n_loc, "query_tokens_per_rank": nq_loc,
                       "order": w.order, "opt": w.opt,
                       "parallelism": f"context parallel over {world} ranks (token slices, one all-reduce "
                                      f"of {cp.buf.nbytes} gradient bytes per update)",
                       "l2": "inputs larger than L2 (no flush)" if h2d >= 2 * L2_BYTES else "L2 not flushed",
                       "launch": "direct calls"},
            "roofline": {"bound": "tensor" if grad["tensor_launches"] > 0 else "alu", "achieved": achieved,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "traffic": None, "kernel": "rank 0's slice gradient", "peak_source": f"dense bf16 burst, {pk_src}",
                         "ms_per_launch": grad_ms, "flop_per_launch": grad_flop},
            "e2e": {"value": tok / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d * world,
                    "d2h_bytes_per_step": ho.numel() * ho.element_size() * world, "ms_per_step": e2e_ms},
            "gpu_launches": launches, "clocks": ck,
            "phases_ms_per_step": {p_: prof[p_]["ms"] / args.steps for p_ in prof}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(w)
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if pg:
        pg.destroy_process_group()
    return 0


def main():
    args = parse()
    w = li.WORKLOADS[args.workload]
    reduced = args.update_tokens is not None or args.query_tokens is not None
    if reduced:
        w = w.with_tokens(args.update_tokens or w.n_kv, n_q=args.query_tokens)
        w = dataclasses.replace(w, name=f"{w.name} (reduced: {w.n_kv} update, {w.n_q} query tokens per head)")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.context_parallel:
        return run_context_parallel(args, w)
    rank, world, local = dist_env()
    import torch
    from chunk_test_step_b300 import lact as L

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg:
            pg.barrier()

    # ---- inputs: generated on the host once, resident in HBM for `value`
    inp = li.make_inputs(w)
    hq, hk, hv, he = pinned_inputs(w, inp)
    q, k, v, e = (x.to(dev, non_blocking=True) for x in (hq, hk, hv, he))
    W1, W2, W3 = (None if x is None else torch.from_numpy(x).to(dev) for x in (inp.W1, inp.W2, inp.W3))
    cfg = L.make_config(w.B, w.H, w.d, w.dh, w.dtype, w.opt, max_chunk=w.chunk, ns_steps=w.ns_steps,
                        ns_a=w.ns_a, ns_b=w.ns_b, ns_c=w.ns_c, muon_lr=w.muon_lr, momentum=w.momentum,
                        memory=w.memory)
    layer = L.LactLayer(cfg, W1, W2, W3, device=dev)
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    def step(s=None):
        L.lact_sequence(layer.handle, order, q, w.n_q, k, v, e, w.n_kv, w.chunk, o, stream if s is None else s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = L.lact_sync_status(layer.handle)
    if st != L.LACT_OK:
        raise RuntimeError(f"device status after warm-up: {L.lact_status_str(st)}")

    # ---- timed regions. Inputs above twice the L2 (126 MB) stream from HBM
    # every step; smaller ones get the L2 flushed (a 256 MB write, untimed)
    # before every step, each step then timed on its own.
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v, e))
    flush = in_bytes < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    def timed_steps(run):
        barrier()
        torch.cuda.synchronize(dev)
        if not flush:
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(args.steps):
                run()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            ms = ev0.elapsed_time(ev1)
        else:
            ms = 0.0
            for _ in range(args.steps):
                scrub.fill_(1.0)
                ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ev0.record(stream)
                run()
                ev1.record(stream)
                torch.cuda.synchronize(dev)
                ms += ev0.elapsed_time(ev1)
        barrier()
        return ms

    # The step as one CUDA graph: lact_sequence captured once (every kernel
    # and stream fork/join of the call becomes a node) and replayed on the
    # timing stream, so the timed region holds no host launch overhead. A
    # replay runs every kernel of the step on the same device buffers, so K
    # replays are K layer steps (the weights move on each); the results equal
    # those of direct calls bit for bit.
    graph, per_step, launch_mode = None, 0, "direct calls"
    if not args.no_graph:
        try:
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            c0 = L.lact_launch_count()
            # thread-local capture: CUDA calls of other host threads (a
            # communicator's watchdog) do not invalidate it
            with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                step(cap)
            per_step = L.lact_launch_count() - c0
            torch.cuda.synchronize(dev)
            graph, launch_mode = g, "one CUDA graph replay per step"
        except RuntimeError as exc:   # capture refused: time direct calls instead, and say so
            torch.cuda.synchronize(dev)
            launch_mode = f"direct calls (graph capture failed: {str(exc).splitlines()[0][:120]})"

    # region 1: the measured value (no per-phase events in the stream)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    n0 = L.lact_launch_count()
    ms_total = max_over_ranks(timed_steps(step if graph is None else graph.replay), pg, dev)
    launches = L.lact_launch_count() - n0 if graph is None else per_step * args.steps
    ck = clocks.stop()
    ms_step = ms_total / args.steps
    tok = tokens_per_step(w)
    value = job_throughput(tok, world, ms_step)
    # region 2: the same steps with the library's CUDA events around every
    # phase, on the launching stream (per-kernel times for the roofline)
    L.lact_set_profiling(layer.handle, True)
    ms_prof = max_over_ranks(timed_steps(step), pg, dev) / args.steps
    prof = L.lact_get_profile(layer.handle)
    L.lact_set_profiling(layer.handle, False)

    # ---- e2e: host (pinned) inputs copied in, the call, the output copied
    # out, every step. Two sets of device buffers: step t+1's inputs are
    # copied in (one copy stream per tensor) while step t computes, and step
    # t's output is copied out beside step t+1. The host link (not the GPU)
    # bounds this, so the overlap hides the compute and the output copy.
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, he))
    d2h = ho.numel() * ho.element_size()
    bufs = [(q, k, v, e, o), tuple(torch.empty_like(x) for x in (q, k, v, e, o))]
    copy_streams = [torch.cuda.Stream(dev) for _ in range(4)]
    out_stream = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    in_ready = [[ev() for _ in range(4)] for _ in range(2)]
    done = [ev(), ev()]
    out_read = [ev(), ev()]   # the output copy of the last step that used the set
    host = (hq, hk, hv, he)

    def copy_in(b, after=None):
        for i, cs in enumerate(copy_streams):
            if after is not None:
                cs.wait_event(after)
            with torch.cuda.stream(cs):
                bufs[b][i].copy_(host[i], non_blocking=True)
            in_ready[b][i].record(cs)

    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_in(0, after=e0)
    for t in range(args.e2e_steps):
        b = t % 2
        if t + 1 < args.e2e_steps:
            # buffer set 1-b is free once step t-1 (which read it) is done
            copy_in(1 - b, after=done[1 - b] if t >= 1 else e0)
        for i in range(4):
            stream.wait_event(in_ready[b][i])
        if t >= 2:
            stream.wait_event(out_read[b])   # step t-2's output is out of the buffer
        bq, bk, bv, be, bo = bufs[b]
        L.lact_sequence(layer.handle, order, bq, w.n_q, bk, bv, be, w.n_kv, w.chunk, bo, stream)
        done[b].record(stream)
        out_stream.wait_event(done[b])
        with torch.cuda.stream(out_stream):
            ho.copy_(bo, non_blocking=True)
        out_read[b].record(out_stream)
    stream.wait_stream(out_stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, pg, dev)
    st = L.lact_sync_status(layer.handle)
    if st != L.LACT_OK:
        raise RuntimeError(f"device status after the timed region: {L.lact_status_str(st)}")

    # ---- roofline of the dominant phase: the chunk gradient (the fused
    # kernel at head dim 128; two kernels per token slice at head dim 256),
    # timed per call with CUDA events on the launching stream
    pk, pk_src = peaks()
    fl = flops(w)
    grad = prof["grad"]
    chunks = 1 if w.order == "set" else -(-w.n_kv // w.chunk)
    grad_ms = grad["ms"] / max(1, grad["calls"])
    grad_flop = fl["update"] / chunks
    achieved = grad_flop / (grad_ms / 1e3) / 1e12
    tensor = grad["tensor_launches"] > 0
    if w.memory == "linear":
        # the linear memory's gradient reads k, v (and eta) once for 2 d^2 FLOP a token: HBM-bound
        esz = 2 if w.dtype == "bf16" else 4
        grad_bytes = w.B * w.H * (w.n_kv / chunks) * (2 * w.d * esz + 4)
        achieved = grad_bytes / (grad_ms / 1e3) / 1e9
        peak, bound, note = pk["hbm_gbs"], "hbm", f"HBM copy bandwidth, {pk_src}"
        kernel = "k_wgrad_tc (linear, -eta V scaled in shared memory)" if tensor else "k_lin_grad_simt"
    elif tensor:
        peak, bound, note = pk["bf16_tflops"], "tensor", f"dense bf16 burst, {pk_src}"
        kernel = "k_grad_tc" if w.d == 128 else "k_fwdbwd_tc + k_wgrad_tc"
    else:
        # the fp32-io path computes in fp64 on the CUDA cores: B300's nominal
        # dense fp64 rate
        peak = FP64_TFLOPS
        bound, note = "alu", "fp64 FMA (the fp32-io path computes in fp64): nominal 1.25 TFLOP/s"
        kernel = "k_grad_simt"
    roof = {"bound": bound, "achieved": achieved, "peak": peak, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": achieved / peak,
            "traffic": measured_traffic(w, reduced), "traffic_unit": "bytes per launch", "kernel": kernel,
            "peak_source": note, "ms_per_launch": grad_ms, "flop_per_launch": grad_flop,
            "launches_per_call": grad["launches"] / max(1, grad["calls"])}
    if bound == "tensor":
        # the same rate against the tensor cores' own dense rate (4,096 bf16
        # MACs per clock per SM) at the maximum and at the sampled SM clock
        for key, mhz in (("max_clock", pk.get("sm_max_mhz", 2032.0)), ("median_clock", (ck or {}).get("sm_mhz"))):
            if mhz:
                p_clk = dense_bf16_tflops(mhz)
                roof["peak_dense_" + key] = p_clk
                roof["frac_dense_" + key] = achieved / p_clk

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d, "dh": w.dh,
                       "update_tokens_per_head": w.n_kv, "query_tokens_per_head": w.n_q,
                       "chunk": w.chunk, "order": w.order, "opt": w.opt,
                       "l2": ("L2 flushed before every step (256 MB write, untimed)" if flush
                              else "inputs larger than L2 (no flush)"),
                       "tflops_per_s": fl["total"] / (ms_step / 1e3) / 1e12 * world,
                       "launch": launch_mode},
            "roofline": roof,
            "e2e": {"value": job_throughput(tok, world, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": launches,
            "clocks": ck,
            "phases_ms_per_step": {p: prof[p]["ms"] / args.steps for p in prof},
            "profiled_ms_per_step": ms_prof}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(w)
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
