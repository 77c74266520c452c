"""Context-parallel update (one chunk cut across ranks by tokens, the slice
gradients summed, one update everywhere): the review page's "Video and
distributed computation".

On CPU: the token partition, and the whole composition on two gloo ranks with
the oracle's gradient and update in place of liblact's (each rank's slice
gradient, one all-reduce, the same step on both ranks), against the oracle's
single-device update on the whole chunk. On the GPU: the liblact phases of
two ranks' slices on one device (two states; the sum the all-reduce would
form taken by hand), against the oracle.
"""
import os
import socket
import sys
from types import SimpleNamespace

import numpy as np
import pytest
import torch.multiprocessing as mp

import lact_inputs as li
from chunk_test_step_b300.context_parallel import TILE, token_range

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("n", [0, 1, 127, 128, 129, 1000, 196608, 5 * 128 + 3])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_token_ranges_cover_the_chunk_once_in_whole_tiles(n, world):
    rs = [token_range(n, r, world) for r in range(world)]
    assert rs[0][0] == 0 and rs[-1][1] == n
    for (a0, a1), (b0, b1) in zip(rs, rs[1:]):
        assert a1 == b0                      # contiguous, in rank order
    sizes = [b - a for a, b in rs]
    assert all(s >= 0 for s in sizes) and sum(sizes) == n
    for a, b in rs:
        assert (a % TILE == 0 or a == n) and (b % TILE == 0 or b == n)
    tiles = [-(-s // TILE) for s in sizes]
    assert max(tiles) - min(tiles) <= 1      # balanced to one tile


def test_token_range_rejects_bad_arguments():
    for args in ((10, 2, 2), (10, -1, 2), (10, 0, 0), (-1, 0, 1)):
        with pytest.raises(ValueError):
            token_range(*args)


# ------------------------------------------------ two gloo ranks, the oracle inside
def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cp_worker(rank, world, port, opt, memory, out, n=1000):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import lact_inputs as li
    from chunk_test_step_b300 import lact as L
    from chunk_test_step_b300.context_parallel import ContextParallelUpdate
    from oracle import lact_oracle as O
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        d, dh = 16, (16 if memory == "linear" else 32)
        w = li.Workload(0, "cp-tiny", 1, 2, d, dh, "f32", "set", opt, n, 40, n, 4321, memory=memory)
        inp = li.make_inputs(w)
        lin = memory == "linear"
        Wh = [inp.W1] if lin else [inp.W1, inp.W2, inp.W3]
        # this rank's state: per (b, h) the head's initial weights (and velocities)
        state = {(b, h): [x[h].astype(np.float64) for x in Wh] for b in range(w.B) for h in range(w.H)}
        mom = {key: O.zero_velocity(Ws) for key, Ws in state.items()}
        kw = dict(lr=w.muon_lr, ns_steps=w.ns_steps, a=w.ns_a, b=w.ns_b, c=w.ns_c)

        def gradient(k, v, eta, n, grads, stream=None):
            for (b, h), Ws in state.items():
                g = O.memory_gradient(Ws, li.as_f64(k[b, h]), li.as_f64(v[b, h]), eta[b, h].astype(np.float64))
                for m, gm in enumerate(g):
                    grads[m][b, h] = torch.from_numpy(gm)

        def step(grads, stream=None):
            for (b, h), Ws in state.items():
                g = [grads[m][b, h].double().numpy() for m in range(len(Ws))]
                if opt == "momentum":
                    for m in range(len(Ws)):
                        mom[(b, h)][m] = O.momentum_velocity(mom[(b, h)][m], g[m], w.momentum)
                    state[(b, h)] = [O.renorm_update(Wm, -M) for Wm, M in zip(Ws, mom[(b, h)])]
                else:
                    state[(b, h)] = [O.renorm_update(Wm, O.optimizer_delta(gm, opt, **kw)) for Wm, gm in zip(Ws, g)]

        cfg = L.make_config(w.B, w.H, d, dh, "f32", opt, max_chunk=w.n_kv, memory=memory)
        # an fp64 buffer: the composition is then exact up to the order of the additions
        cp = ContextParallelUpdate(SimpleNamespace(cfg=cfg, handle=None), device="cpu", gradient=gradient, step=step,
                                   dtype=torch.float64)
        assert (cp.rank, cp.world) == (rank, world)
        for _ in range(2):                     # two chunks: the state carries across them
            t0, t1 = cp.slice(w.n_kv)
            cp.update(inp.k[:, :, t0:t1], inp.v[:, :, t0:t1], inp.eta[:, :, t0:t1], t1 - t0)
        # the oracle on one device: two whole-chunk updates on the same tokens
        worst = 0.0
        for (b, h), Ws in state.items():
            W0 = tuple(x[h].astype(np.float64) for x in Wh)
            K, V, e = li.as_f64(inp.k[b, h]), li.as_f64(inp.v[b, h]), inp.eta[b, h].astype(np.float64)
            mom_ref = O.zero_velocity(W0) if opt == "momentum" else None
            Wr = O.chunk_update(W0, K, V, e, opt, mom=mom_ref, beta=w.momentum, **kw)
            Wr = O.chunk_update(Wr, K, V, e, opt, mom=mom_ref, beta=w.momentum, **kw)
            for a, r in zip(Ws, Wr):
                worst = max(worst, float(np.linalg.norm(a - r) / np.linalg.norm(r)))
        # every rank holds the same weights
        flat = torch.from_numpy(np.concatenate([x.ravel() for Ws in state.values() for x in Ws]))
        other = flat.clone()
        dist.broadcast(other, src=0)
        out.put((rank, worst, bool(torch.equal(flat, other)), cp.buf.nbytes))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("opt,memory,world,n", [("gd", "swiglu", 2, 1000), ("muon", "swiglu", 2, 1000),
                                                ("momentum", "swiglu", 2, 1000), ("muon", "linear", 2, 1000),
                                                ("gd", "swiglu", 3, 300)])
def test_gloo_ranks_sum_slice_gradients_into_the_whole_chunk_update(opt, memory, world, n):
    # (three ranks on 300 tokens: slices of 128, 128 and 44 tokens; the
    # uneven, ragged last slice still sums to the whole chunk)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_worker, args=(r, world, port, opt, memory, q, n)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    d, dh = 16, (16 if memory == "linear" else 32)
    for rank, worst, same, nbytes in res:
        assert worst < 1e-10, (rank, worst)     # fp64: only the order of the additions differs
        assert same, rank
        # the exchange: 3 d dh fp32 per (b, h) (d d for the linear memory), 2 heads
        assert nbytes == 2 * 8 * (d * d if memory == "linear" else 3 * d * dh)   # (fp64 here, fp32 in use)


# ------------------------------------------------ the liblact phases on the GPU
@pytest.mark.gpu
@pytest.mark.parametrize("num", [4, 2, 10, 7])
def test_two_slices_on_the_gpu_match_the_whole_chunk(num):
    import torch
    from chunk_test_step_b300 import lact as L
    from chunk_test_step_b300.context_parallel import ContextParallelUpdate
    from oracle import lact_oracle as O
    from tests.harness import (TOL, compare_change, config_for, dw_tol, initial_weights, max_rel_l2_per_head,
                               record, to_device, to_host_f64)
    w = li.WORKLOADS[num].with_tokens(3 * 1024 + 77, seed=li.WORKLOADS[num].seed + 6000)
    inp = li.make_inputs(w)
    world = 2
    ranks = []
    for r in range(world):
        layer = L.LactLayer(config_for(w, max_chunk=w.n_kv), to_device(inp.W1), to_device(inp.W2), to_device(inp.W3))
        cp = ContextParallelUpdate(layer)
        cp.rank, cp.world = r, world           # two ranks' slices, on one device
        t0, t1 = cp.slice(w.n_kv)
        sl = [to_device(np.ascontiguousarray(x[:, :, t0:t1])) for x in (inp.k, inp.v, inp.eta)]
        cp.compute_gradient(*sl, t1 - t0)
        ranks.append((layer, cp))
    total = sum(cp.buf.flat for _, cp in ranks)     # what the all-reduce (sum) forms
    for layer, cp in ranks:
        cp.buf.flat.copy_(total)
        cp.step()
    Ws = [[x for x in layer.weights() if x is not None] for layer, _ in ranks]
    torch.cuda.synchronize()
    for a, b in zip(*Ws):
        assert torch.equal(a, b)
    got = [to_host_f64(x) for x in Ws[0]]
    W0 = initial_weights(w, inp)
    mats = (inp.W1,) if w.memory == "linear" else (inp.W1, inp.W2, inp.W3)
    want = [np.zeros_like(g) for g in got]
    for b in range(w.B):
        for h in range(w.H):
            W0h = tuple(x[h].astype(np.float64) for x in mats)
            Wf = O.chunk_update(W0h, li.as_f64(inp.k[b, h]), li.as_f64(inp.v[b, h]),
                                inp.eta[b, h].astype(np.float64), w.opt, lr=w.muon_lr, ns_steps=w.ns_steps,
                                mom=O.zero_velocity(W0h) if w.opt == "momentum" else None, beta=w.momentum)
            for m in range(len(got)):
                want[m][b, h] = Wf[m]
    for m in range(len(got)):
        err = record("context_parallel_2_slices", w, "W%d" % (m + 1), max_rel_l2_per_head(got[m], want[m]),
                     TOL[w.dtype])
        assert err < TOL[w.dtype], (m, err)
    dW = compare_change(w, W0[:len(got)], got, want, exact_gradient=False, test="context_parallel_2_slices")
    assert max(dW.values()) < dw_tol(w, False), dW
    for layer, _ in ranks:
        layer.close()


def _cp_empty_worker(rank, world, port, out):
    # more ranks than tiles: the ranks past the last tile hold an empty slice
    # and contribute zeros; everyone still ends with the whole chunk's update
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import lact_inputs as li
    from chunk_test_step_b300 import lact as L
    from chunk_test_step_b300.context_parallel import ContextParallelUpdate
    from oracle import lact_oracle as O
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        d, dh, n = 16, 32, 150                          # 2 tiles of 128 tokens over 4 ranks
        w = li.Workload(0, "cp-empty", 1, 1, d, dh, "f32", "set", "gd", n, 8, n, 4322)
        inp = li.make_inputs(w)
        W = [x[0].astype(np.float64) for x in (inp.W1, inp.W2, inp.W3)]

        def gradient(k, v, eta, n_local, grads, stream=None):
            if n_local == 0:
                for g in grads[:3]:
                    g.zero_()
                return
            for m, gm in enumerate(O.chunk_gradient(*W, li.as_f64(k[0, 0]), li.as_f64(v[0, 0]),
                                                    eta[0, 0].astype(np.float64))):
                grads[m][0, 0] = torch.from_numpy(gm)

        result = {}

        def step(grads, stream=None):
            result["W"] = [O.renorm_update(Wm, -grads[m][0, 0].double().numpy()) for m, Wm in enumerate(W)]

        cfg = L.make_config(1, 1, d, dh, "f32", "gd", max_chunk=n)
        cp = ContextParallelUpdate(SimpleNamespace(cfg=cfg, handle=None), device="cpu", gradient=gradient, step=step,
                                   dtype=torch.float64)
        t0, t1 = cp.slice(n)
        cp.update(inp.k[:, :, t0:t1], inp.v[:, :, t0:t1], inp.eta[:, :, t0:t1], t1 - t0)
        want = O.chunk_update(tuple(W), li.as_f64(inp.k[0, 0]), li.as_f64(inp.v[0, 0]),
                              inp.eta[0, 0].astype(np.float64), "gd")
        err = max(float(np.linalg.norm(a - b) / np.linalg.norm(b)) for a, b in zip(result["W"], want))
        out.put((rank, t1 - t0, err))
    finally:
        dist.destroy_process_group()


def test_ranks_beyond_the_last_tile_contribute_nothing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_cp_empty_worker, args=(r, 4, port, q)) for r in range(4)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert [r[1] for r in res] == [128, 22, 0, 0]
    assert all(r[2] < 1e-12 for r in res), res
