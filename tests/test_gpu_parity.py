"""GPU parity: liblact (through its C ABI) against the fp64 oracle on the same
seeded inputs. Max relative L2 error per tensor per (b, h) must stay within
1e-4 for fp32 workloads and 2e-2 for bf16 workloads.

Sizes span several tiles with ragged tails; each row of the hot path
(readout, chunk gradient, optimiser + renorm) is also checked on its own.
"""
import dataclasses

import numpy as np
import pytest

import lact_inputs as li
from oracle import lact_oracle as O
from tests.harness import (TOL, compare, compare_change, config_for, dw_tol, initial_weights, max_rel_l2_per_head,
                           record, rel_l2, run_gpu, to_device, to_host_f64)

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    assert torch.cuda.is_available()
    return torch


def _layer(w, inp, max_chunk=None):
    from chunk_test_step_b300 import lact as L
    return L.LactLayer(config_for(w, max_chunk), to_device(inp.W1), to_device(inp.W2), to_device(inp.W3))


# Reduced token counts of each workload: several tiles and a ragged tail.
SMALL = {
    1: dict(n_kv=2048),                       # the whole tiny workload
    2: dict(n_kv=2 * 2048 + 301),             # two full chunks + a partial one
    3: dict(n_kv=2048),
    4: dict(n_kv=5000 + 13, n_q=333),
    5: dict(n_kv=8192 + 77, n_q=500),
    6: dict(n_kv=2048),                       # the whole tiny momentum workload
    7: dict(n_kv=2 * 2048 + 301),
    8: dict(n_kv=4096 + 1000),                # one full chunk + a partial one
    9: dict(n_kv=2048),                       # the whole tiny linear workload
    10: dict(n_kv=5000 + 13, n_q=333),
}


def _small(num):
    w = li.WORKLOADS[num]
    return w.with_tokens(seed=w.seed + 1000, **SMALL[num])


# ------------------------------------------------------------- row a1: readout
@pytest.mark.parametrize("num,n_q", [(1, None), (2, None), (4, None), (5, 1), (5, 127), (5, 128 * 9 + 3)])
def test_apply_matches_oracle(num, n_q):
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = _small(num)
    if n_q is not None:
        w = w.with_tokens(w.n_kv, n_q=n_q)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    q = to_device(inp.q)
    o = torch.empty_like(q)
    L.lact_chunk_apply(layer.handle, q, w.n_q, o)
    got = to_host_f64(o)
    want = np.zeros_like(got)
    for b in range(w.B):
        for h in range(w.H):
            want[b, h] = O.fast_weight_apply(inp.W1[h].astype(np.float64), inp.W2[h].astype(np.float64),
                                             inp.W3[h].astype(np.float64), li.as_f64(inp.q[b, h]))
    err = record("apply", w, "o", max_rel_l2_per_head(got, want), TOL[w.dtype])
    assert err < TOL[w.dtype], err


# ---------------------------------------------------- rows a2-a4: gradient
def _check_gradient(w, test="chunk_gradient"):
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    n = w.n_kv
    inp = li.make_inputs(w)
    layer = _layer(w, inp, max_chunk=n)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    g = [torch.empty(w.B, w.H, *s, device="cuda") for s in ((w.dh, w.d), (w.d, w.dh), (w.dh, w.d))]
    L.lact_chunk_gradient(layer.handle, k, v, e, n, *g)
    got = [to_host_f64(x) for x in g]
    worst = [0.0, 0.0, 0.0]
    for b in range(w.B):
        for h in range(w.H):
            want = O.chunk_gradient(inp.W1[h].astype(np.float64), inp.W2[h].astype(np.float64),
                                    inp.W3[h].astype(np.float64), li.as_f64(inp.k[b, h]),
                                    li.as_f64(inp.v[b, h]), inp.eta[b, h].astype(np.float64))
            for m in range(3):
                err = rel_l2(got[m][b, h], want[m])
                worst[m] = max(worst[m], err)
                assert err < TOL[w.dtype], (m, b, h, err)
    for m in range(3):
        record(test, w, "gW%d" % (m + 1), worst[m], TOL[w.dtype])


@pytest.mark.parametrize("num,n", [(1, 1000 + 37), (2, 2048 + 5), (4, 4096 + 99), (5, 3 * 128 + 1),
                                   (4, 1), (4, 127), (5, 128), (5, 37 * 128 + 5), (2, 1), (2, 129)])
def test_chunk_gradient_matches_oracle(num, n):
    _check_gradient(li.WORKLOADS[num].with_tokens(n, seed=li.WORKLOADS[num].seed + 2000))


def test_gradient_at_head_dim_256_spans_several_token_slices():
    # head dim 256 takes the gradient per 4,096-token slice (two kernels per
    # slice, the GEMMs adding into the result): three slices, the last ragged
    w = dataclasses.replace(li.WORKLOADS[2], H=1)
    _check_gradient(w.with_tokens(2 * 4096 + 77, seed=w.seed + 2100), "chunk_gradient_d256_slices")


# ------------------------------------------------ linear fast-weight memory
@pytest.mark.parametrize("num,n", [(9, 1000 + 37), (10, 4096 + 99), (10, 1), (10, 64 * 37 + 5), (9, 1)])
def test_linear_chunk_gradient_matches_oracle(num, n):
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(n, seed=li.WORKLOADS[num].seed + 2200)
    inp = li.make_inputs(w)
    layer = _layer(w, inp, max_chunk=n)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    g = torch.empty(w.B, w.H, w.d, w.d, device="cuda")
    L.lact_chunk_gradient(layer.handle, k, v, e, n, g, None, None)
    got = to_host_f64(g)
    for b in range(w.B):
        for h in range(w.H):
            want = O.linear_chunk_gradient(inp.W1[h].astype(np.float64), li.as_f64(inp.k[b, h]),
                                           li.as_f64(inp.v[b, h]), inp.eta[b, h].astype(np.float64))
            err = record("linear_chunk_gradient", w, "gW", rel_l2(got[b, h], want), TOL[w.dtype], b=b, h=h)
            assert err < TOL[w.dtype], (b, h, err)


@pytest.mark.parametrize("num,n_q", [(9, 2048), (10, 333), (10, 1), (10, 128 * 5)])
def test_linear_apply_matches_oracle(num, n_q):
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(128, n_q=n_q, seed=li.WORKLOADS[num].seed + 2300)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    q = to_device(inp.q)
    o = torch.empty_like(q)
    L.lact_chunk_apply(layer.handle, q, w.n_q, o)
    got = to_host_f64(o)
    for b in range(w.B):
        for h in range(w.H):
            want = O.linear_apply(inp.W1[h].astype(np.float64), li.as_f64(inp.q[b, h]))
            err = record("linear_apply", w, "o", rel_l2(got[b, h], want), TOL[w.dtype], b=b, h=h)
            assert err < TOL[w.dtype], (b, h, err)


# ------------------------------------------- rows a5-a7: optimiser + renorm
# (workload, update rule, Newton-Schulz steps). Few-step Muon cases bind each
# GEMM of the Newton-Schulz kernels tightly (the drift from accumulation order
# stays near 1e-5 there); the five-step cases are the layers' own setting.
APPLY_GRADIENT_CASES = [(1, "gd", 5), (2, "gd", 5), (7, "momentum", 5), (3, "muon", 5), (3, "muon", 1),
                        (4, "muon", 5), (4, "muon", 1), (4, "muon", 2), (4, "muon", 3), (5, "muon", 5),
                        (8, "muon", 5), (8, "muon", 2), (10, "muon", 5), (10, "muon", 1), (10, "muon", 2)]


@pytest.mark.parametrize("num,opt,ns_steps", APPLY_GRADIENT_CASES)
def test_apply_gradient_matches_oracle(num, opt, ns_steps):
    # optimiser step + row renorm from a gradient given exactly to both sides:
    # the new weights within the weight budget, the CHANGE of the weights
    # within dw_tol (the only path from the gradient to the weights here is
    # the update rule: the Newton-Schulz kernel for Muon)
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(128, seed=li.WORKLOADS[num].seed + 3000, opt=opt, ns_steps=ns_steps)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    # gradients drawn by the generator at the scale of real chunk gradients
    s = w.seed + 3000
    shapes = ((w.d, w.d),) if w.memory == "linear" else ((w.dh, w.d), (w.d, w.dh), (w.dh, w.d))
    G = [li.normal(s, 20 + m, (w.B, w.H) + sh, scale=0.05) for m, sh in enumerate(shapes)]
    L.lact_apply_gradient(layer.handle, *(to_device(x) for x in G), *([None] * (3 - len(G))))
    got = layer.weights()
    torch.cuda.synchronize()
    got = [to_host_f64(x) for x in got if x is not None]
    W0 = initial_weights(w, inp)[:len(G)]
    want = [np.zeros_like(g) for g in got]
    for b in range(w.B):
        for h in range(w.H):
            for m in range(len(G)):
                g = G[m][b, h].astype(np.float64)
                delta = -g if opt == "momentum" else O.optimizer_delta(g, opt, lr=w.muon_lr, ns_steps=ns_steps)
                want[m][b, h] = O.renorm_update(W0[m][b, h], delta)
                # row norms are those before the update
                np.testing.assert_allclose(np.linalg.norm(got[m][b, h], axis=1),
                                           np.linalg.norm(W0[m][b, h], axis=1), rtol=2e-6)
    test = "apply_gradient"
    for m in range(len(G)):
        err = record(test, w, "W%d" % (m + 1), max_rel_l2_per_head(got[m], want[m]), TOL[w.dtype])
        assert err < TOL[w.dtype], (m, err)
    dW = compare_change(w, W0, got, want, exact_gradient=True, test=test)
    assert max(dW.values()) < dw_tol(w, True), dW


@pytest.mark.parametrize("num", [6, 7])
def test_momentum_velocity_carries_across_two_steps(num):
    # two optimiser steps from given gradients: the second moves by
    # beta * (first gradient) + (second gradient), then renorm
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(128, seed=li.WORKLOADS[num].seed + 3100)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    shapes = ((w.dh, w.d), (w.d, w.dh), (w.dh, w.d))
    s = w.seed + 3100
    G = [[li.normal(s, 30 + 3 * k + m, (w.B, w.H) + sh, scale=0.05) for m, sh in enumerate(shapes)] for k in range(2)]
    for k in range(2):
        L.lact_apply_gradient(layer.handle, *(to_device(x) for x in G[k]))
    got = [to_host_f64(x) for x in layer.weights()]
    torch.cuda.synchronize()
    W0 = (inp.W1, inp.W2, inp.W3)
    for b in range(w.B):
        for h in range(w.H):
            for m in range(3):
                M = O.momentum_velocity(np.zeros(shapes[m]), G[0][m][b, h].astype(np.float64), w.momentum)
                Wm = O.renorm_update(W0[m][h].astype(np.float64), -M)
                M = O.momentum_velocity(M, G[1][m][b, h].astype(np.float64), w.momentum)
                Wm = O.renorm_update(Wm, -M)
                err = record("momentum_two_steps", w, "W%d" % (m + 1), rel_l2(got[m][b, h], Wm), TOL[w.dtype], b=b, h=h)
                assert err < TOL[w.dtype], (m, b, h, err)
                dchg = record("momentum_two_steps", w, "dW%d" % (m + 1),
                              rel_l2(got[m][b, h] - W0[m][h], Wm - W0[m][h]), dw_tol(w, True), kind="change", b=b, h=h)
                assert dchg < dw_tol(w, True), (m, b, h, dchg)


# ------------------------------------------------- whole layer calls (a8)
def _check_sequence(w, test):
    inp = li.make_inputs(w)
    got = run_gpu(w, inp)
    want = O.run_workload(w, inp)
    errs = compare(w, got, want, test)
    assert max(errs.values()) < TOL[w.dtype], errs
    # the change of the weights over the call, against its own budget
    dW = compare_change(w, initial_weights(w, inp), got[1:], want[1:], exact_gradient=False, test=test)
    assert max(dW.values()) < dw_tol(w, False), dW


@pytest.mark.parametrize("num", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10])
def test_sequence_matches_oracle(num):
    _check_sequence(_small(num), "sequence")


@pytest.mark.parametrize("num", [4, 5, 8, 10])
def test_muon_sequence_with_two_newton_schulz_steps(num):
    # With two Newton-Schulz steps the update barely amplifies the gradient's
    # bf16 rounding, so the change of the weights over a whole layer call is
    # held to the bf16 budget: the gradient, Newton-Schulz, update and renorm
    # kernels all bind.
    _check_sequence(_small(num).with_tokens(_small(num).n_kv, ns_steps=2), "sequence_ns2")


def test_set_mode_slices_sum_before_one_step():
    w = li.WORKLOADS[4].with_tokens(3000, n_q=100, seed=77)
    w = dataclasses.replace(w, chunk=1024)
    inp = li.make_inputs(w)
    got = run_gpu(w, inp)
    want = O.run_workload(w, inp)   # set mode: one step on all 3000 tokens
    errs = compare(w, got, want, "set_slices")
    assert max(errs.values()) < TOL[w.dtype], errs


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("opt", ["gd", "muon"])
def test_empty_update_leaves_weights(opt):
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[1].with_tokens(64, opt=opt)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    z = torch.zeros(16, device="cuda")
    L.lact_chunk_update(layer.handle, z, z, z, 0)
    L.lact_chunk_apply(layer.handle, z, 0, z)
    got = [to_host_f64(x) for x in layer.weights()]
    torch.cuda.synchronize()
    for m, W0 in enumerate((inp.W1, inp.W2, inp.W3)):
        np.testing.assert_array_equal(got[m][0], W0.astype(np.float64))
    assert L.lact_sync_status(layer.handle) == L.LACT_OK


def test_update_beyond_max_chunk_is_rejected():
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[1].with_tokens(64)
    inp = li.make_inputs(w)
    layer = _layer(w, inp, max_chunk=64)
    k = torch.zeros(1, 2, 65, 64, device="cuda")
    e = torch.zeros(1, 2, 65, device="cuda")
    with pytest.raises(L.LactError) as ex:
        L.lact_chunk_update(layer.handle, k, k, e, 65)
    assert ex.value.status == L.LACT_ERR_INVALID_ARG


@pytest.mark.parametrize("num", [3, 2, 6, 7, 9, 10])
def test_checkpoint_resume_equals_one_run(num):
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    # (the set-mode workloads' shapes run here in the causal order)
    w = li.WORKLOADS[num].with_tokens(1024, n_q=1024, chunk=256)
    inp = li.make_inputs(w)
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    one = _layer(w, inp)
    o_one = one.sequence(L.LACT_CAUSAL_APPLY_THEN_UPDATE, q, k, v, e, 256)
    W_one = one.weights()
    # first half, export, a fresh state imports, second half
    a = _layer(w, inp)
    qa, ka, va, ea = (x[:, :, :512].contiguous() for x in (q, k, v, e))
    o_a = a.sequence(L.LACT_CAUSAL_APPLY_THEN_UPDATE, qa, ka, va, ea, 256)
    saved = torch.empty(L.lact_state_bytes(a.handle), dtype=torch.uint8, device="cuda")
    L.lact_export_state(a.handle, saved)
    b = _layer(w, inp)
    L.lact_import_state(b.handle, saved)
    qb, kb, vb, eb = (x[:, :, 512:].contiguous() for x in (q, k, v, e))
    o_b = b.sequence(L.LACT_CAUSAL_APPLY_THEN_UPDATE, qb, kb, vb, eb, 256)
    W_two = b.weights()
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([o_a, o_b], dim=2), o_one)
    for x, y in zip(W_one, W_two):
        assert (x is None and y is None) or torch.equal(x, y)


def test_nonfinite_row_sets_status():
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[1].with_tokens(64)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    W1, W2, W3 = layer.weights()
    W1[0, 0, 3, 5] = float("nan")
    L.lact_set_weights(layer.handle, W1, W2, W3)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    L.lact_chunk_update(layer.handle, k, v, e, 64)
    assert L.lact_sync_status(layer.handle) == L.LACT_ERR_NONFINITE


def test_profiling_counts_phases():
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = _small(5)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    L.lact_set_profiling(layer.handle, True)
    n0 = L.lact_launch_count()
    layer.sequence(L.LACT_SET_UPDATE_THEN_APPLY, q, k, v, e, w.chunk)
    prof = L.lact_get_profile(layer.handle)
    n1 = L.lact_launch_count()
    assert all(prof[p]["calls"] == 1 for p in ("apply", "grad", "ns"))
    # a Muon step whose Newton-Schulz runs on the tensor cores applies the
    # update + renorm in the same kernel: no update launch
    assert prof["update"]["calls"] == 0
    # the split-K sum is its own phase, or (few token splits before a Muon
    # step) done by Newton-Schulz as it reads the partial sums
    assert prof["reduce"]["calls"] in (0, 1)
    assert sum(prof[p]["launches"] for p in prof) == n1 - n0
    assert all(prof[p]["ms"] > 0 for p in prof if prof[p]["calls"] > 0)


@pytest.mark.parametrize("num", [2, 4, 5, 7, 8, 10])
def test_bf16_workloads_run_on_tensor_core_kernels(num):
    # every launch of the readout and gradient phases of the bf16 layers is a
    # tcgen05 kernel (no CUDA-core stand-in)
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = _small(num)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    L.lact_set_profiling(layer.handle, True)
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    layer.sequence(order, q, k, v, e, w.chunk)
    prof = L.lact_get_profile(layer.handle)
    for ph in ("apply", "grad"):
        assert prof[ph]["launches"] > 0 and prof[ph]["tensor_launches"] == prof[ph]["launches"], (ph, prof[ph])


# ------------------------------------------------------ failure detection
def test_bounded_wait_times_out_and_the_state_recovers():
    # a device-side wait that nothing satisfies gives up after its budget,
    # sets the sticky status and returns; after the caller clears it, the
    # same state computes correctly again
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[2].with_tokens(2048 + 300, seed=li.WORKLOADS[2].seed + 5000)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    L.lact_selftest_timeout(layer.handle, 2_000_000)        # 2 ms
    assert L.lact_sync_status(layer.handle) == L.LACT_ERR_TIMEOUT
    L.lact_clear_status(layer.handle)
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    o = layer.sequence(order, q, k, v, e, w.chunk)
    W = layer.weights()
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    errs = compare(w, tuple(to_host_f64(x) for x in (o, *W)), O.run_workload(w, inp), "after_timeout")
    assert max(errs.values()) < TOL[w.dtype], errs


# --------------------------------------------- writes stay inside buffers
@pytest.mark.parametrize("num", [1, 2, 5, 8, 10])
def test_kernels_write_only_inside_their_buffers(num):
    # outputs and the workspace sit between canary regions; after a layer
    # call and a gradient call every canary byte is unchanged
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = _small(num)
    inp = li.make_inputs(w)
    cfg = config_for(w)
    G = 4096                                                  # guard bytes on each side (256-aligned)
    canary = 0xA5

    def guarded(nbytes):
        buf = torch.full((nbytes + 2 * G,), canary, dtype=torch.uint8, device="cuda")
        return buf, buf[G:G + nbytes]

    ws_buf, ws = guarded(L.lact_workspace_bytes(cfg))
    st = L.lact_init_state(cfg, ws, *(to_device(x) for x in (inp.W1, inp.W2, inp.W3)))
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    o_buf, o_bytes = guarded(q.numel() * q.element_size())
    o = o_bytes.view(q.dtype).view(q.shape)
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    L.lact_sequence(st, order, q, w.n_q, k, v, e, w.n_kv, w.chunk, o)
    n = min(w.n_kv, w.chunk)
    shapes = ((w.dh, w.d),) if w.memory == "linear" else ((w.dh, w.d), (w.d, w.dh), (w.dh, w.d))
    gbufs, gs = [], []
    for sh in shapes:
        b, g = guarded(w.B * w.H * sh[0] * sh[1] * 4)
        gbufs.append(b)
        gs.append(g.view(torch.float32))
    gs += [None] * (3 - len(gs))
    L.lact_chunk_gradient(st, k, v, e, n, *gs)
    torch.cuda.synchronize()
    assert L.lact_sync_status(st) == L.LACT_OK
    for buf in [ws_buf, o_buf] + gbufs:
        assert torch.all(buf[:G] == canary) and torch.all(buf[-G:] == canary)
    L.lact_free_state(st)


# ------------------------------------------------- CUDA-graph capture of a step
@pytest.mark.parametrize("num", [1, 2, 5, 8, 10])
def test_sequence_replayed_from_a_cuda_graph_matches_direct_calls(num):
    # lact_sequence captured once into a CUDA graph (side-stream fork/join
    # included) and replayed gives the same outputs and weights, bit for bit,
    # as a direct call from the same starting weights
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = _small(num)
    inp = li.make_inputs(w)
    layer = _layer(w, inp)
    W0 = [None if x is None else to_device(x).unsqueeze(0).repeat(w.B, 1, 1, 1).contiguous()
          for x in (inp.W1, inp.W2, inp.W3)]
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    o = torch.empty_like(q)
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    s = torch.cuda.Stream()

    def step(stream):
        L.lact_sequence(layer.handle, order, q, w.n_q, k, v, e, w.n_kv, w.chunk, o, stream)

    def run(fn):
        with torch.cuda.stream(s):
            L.lact_set_weights(layer.handle, *W0, s)
            fn()
            out = [o.clone()] + [x.clone() for x in layer.weights(s) if x is not None]
        torch.cuda.synchronize()
        return out

    direct = run(lambda: step(s))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    torch.cuda.synchronize()
    replay = run(lambda: g.replay())
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    for a, b in zip(direct, replay):
        assert torch.equal(a, b)
    # and the replay is correct, not merely repeatable
    errs = compare(w, tuple(None if x is None else to_host_f64(x) for x in replay + [None] * (4 - len(replay))),
                   O.run_workload(w, inp), "graph_replay")
    assert max(errs.values()) < TOL[w.dtype], errs


# (workload, tokens, heads): the token splits the gradient picks here are 3
# (workload 4, and 8 at 4,096 tokens), 2 (5), 4 (4 heads of workload 4 at
# 3,072 tokens) and 1 (workload 8 at 256 tokens): Newton-Schulz reads that many
# partial slots, in rounds of pieces whose depth depends on the count
@pytest.mark.parametrize("num,n,heads", [(4, 5000 + 13, None), (8, 4096, None), (5, 8192 + 77, None), (10, 3000, None),
                                         (4, 3072, 4), (8, 256, None)])
def test_update_equals_gradient_then_apply_gradient(num, n, heads):
    # One update (gradient, its split-K sum, Muon step, renorm) against the
    # same done as two calls: lact_chunk_gradient (the sum by the reduction
    # kernel) then lact_apply_gradient. With few token splits the update lets
    # Newton-Schulz add the partial sums as it reads them, in the reduction's
    # order, so the two agree bit for bit either way.
    torch = _torch()
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(n, seed=li.WORKLOADS[num].seed + 7000)
    if heads is not None:
        w = dataclasses.replace(w, H=heads)
    inp = li.make_inputs(w)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    one = _layer(w, inp, max_chunk=n)
    L.lact_set_profiling(one.handle, True)
    L.lact_chunk_update(one.handle, k, v, e, n)
    if heads is not None or n == 256:
        # the cases picked for their 4 and 1 token splits: Newton-Schulz added
        # the slots itself (no reduction launch)
        assert L.lact_get_profile(one.handle)["reduce"]["calls"] == 0
    two = _layer(w, inp, max_chunk=n)
    shapes = ((w.d, w.d),) if w.memory == "linear" else ((w.dh, w.d), (w.d, w.dh), (w.dh, w.d))
    g = [torch.empty(w.B, w.H, *s, device="cuda") for s in shapes] + [None] * (3 - len(shapes))
    L.lact_chunk_gradient(two.handle, k, v, e, n, *g)
    L.lact_apply_gradient(two.handle, *g)
    a, b = one.weights(), two.weights()
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert (x is None and y is None) or torch.equal(x, y)
