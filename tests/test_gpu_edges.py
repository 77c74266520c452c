"""Degenerate cases and the corners of the configuration space, on the GPU
through the C ABI, against the fp64 oracle.

* A weight row of zeros keeps norm zero through an update (renorm scales each
  row back to its pre-update norm, here 0), and the rest follows the oracle.
* All learning rates zero: the chunk gradient is zero, so the weights come
  out bit for bit as they went in (GD, momentum and Muon alike).
* The largest and smallest head and hidden sizes the interface accepts, in
  both io dtypes, through whichever kernels serve them (tensor-core or
  CUDA-core gradient and readout, Newton-Schulz on the tensor cores or, for
  shapes it does not serve, on the CUDA cores).
* A set-order call with no update tokens reads the initial memory and leaves
  it bit for bit; one with no queries still updates.
* Two states driven on two streams at once give what they give one after the
  other (each state owns its workspace and side stream).
"""
import dataclasses

import numpy as np
import pytest

import lact_inputs as li
from oracle import lact_oracle as O
from tests.harness import (TOL, compare, compare_change, config_for, dw_tol, initial_weights, record, run_gpu,
                           to_device, to_host_f64)

pytestmark = pytest.mark.gpu


def _layer(w, inp, max_chunk=None):
    from chunk_test_step_b300 import lact as L
    return L.LactLayer(config_for(w, max_chunk), to_device(inp.W1), to_device(inp.W2), to_device(inp.W3))


@pytest.mark.parametrize("num,mat", [(4, 0), (1, 0), (4, 1), (8, 1)])
def test_zero_weight_row_stays_zero(num, mat):
    # mat 0: a row of W1 (for Muon on the tensor cores a column of Newton-Schulz's
    # tall X, normed over the lanes); mat 1: a row of W2 (a row of the wide X,
    # normed across the cluster's CTAs)
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(1000 + 37, seed=li.WORKLOADS[num].seed + 8000)
    inp = li.make_inputs(w)
    Wz = (inp.W1 if mat == 0 else inp.W2).copy()
    Wz[:, 5, :] = 0.0                       # row 5 of every head's matrix: zeros
    inp = dataclasses.replace(inp, **{"W1" if mat == 0 else "W2": Wz})
    n = w.n_kv
    layer = _layer(w, inp, max_chunk=n)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    L.lact_chunk_update(layer.handle, k, v, e, n)
    got = [to_host_f64(x) for x in layer.weights()]
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    assert np.all(got[mat][:, :, 5, :] == 0.0)
    for b in range(w.B):
        for h in range(w.H):
            Wf = O.chunk_update(tuple(x[h].astype(np.float64) for x in (inp.W1, inp.W2, inp.W3)),
                                li.as_f64(inp.k[b, h]), li.as_f64(inp.v[b, h]), inp.eta[b, h].astype(np.float64),
                                w.opt, lr=w.muon_lr, ns_steps=w.ns_steps)
            assert np.all(Wf[mat][5] == 0.0)
            for m in range(3):
                err = np.linalg.norm(got[m][b, h] - Wf[m]) / np.linalg.norm(Wf[m])
                record("zero_row", w, "W%d" % (m + 1), err, TOL[w.dtype], b=b, h=h)
                assert err < TOL[w.dtype], (m, b, h, err)


@pytest.mark.parametrize("num,opt", [(4, "muon"), (2, "gd"), (7, "momentum"), (3, "muon"), (10, "muon")])
def test_zero_learning_rates_leave_weights_unchanged(num, opt):
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(700 + 3, seed=li.WORKLOADS[num].seed + 8100, opt=opt)
    inp = li.make_inputs(w)
    inp = dataclasses.replace(inp, eta=np.zeros_like(inp.eta))
    layer = _layer(w, inp, max_chunk=w.n_kv)
    before = [None if x is None else x.clone() for x in layer.weights()]
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    L.lact_chunk_update(layer.handle, k, v, e, w.n_kv)
    after = layer.weights()
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    for x, y in zip(before, after):
        assert (x is None and y is None) or torch.equal(x, y)


# (head dim, hidden, io dtype, rule): the largest hidden size (1024) at both
# head dims of the tensor-core path and on the CUDA cores, the smallest head
# dim and hidden size, and Muon where Newton-Schulz runs on the CUDA cores
# (short side 256, or long side above 512).
CORNERS = [
    (128, 1024, "bf16", "muon"),
    (256, 512, "bf16", "muon"),
    (256, 1024, "bf16", "gd"),
    (64, 64, "bf16", "momentum"),
    (32, 128, "bf16", "gd"),
    (32, 64, "f32", "muon"),
    (256, 1024, "f32", "gd"),
    (128, 1024, "f32", "muon"),
    # Newton-Schulz on the tensor cores with the update inside, at the other
    # long sides it serves: n = 256 (one 256-column CTA), n = 384 (a cluster
    # of three 128-column CTAs), and W1/W3 wide with W2 tall (d > dh)
    (128, 256, "bf16", "muon"),
    (128, 384, "bf16", "muon"),
    (256, 128, "bf16", "muon"),
    # the tensor-core path's smallest hidden sizes: two blocks of 64 with all
    # three Newton-Schulz matrices square, and a single block
    (128, 128, "bf16", "muon"),
    (128, 64, "bf16", "gd"),
]


@pytest.mark.parametrize("d,dh,dtype,opt", CORNERS)
def test_configuration_corners_match_oracle(d, dh, dtype, opt):
    base = li.WORKLOADS[1] if dtype == "f32" else li.WORKLOADS[2]
    n = 2 * 256 + 77                        # two causal chunks of 256 and a ragged one
    w = dataclasses.replace(base, name=f"corner-d{d}-dh{dh}-{dtype}-{opt}", B=1, H=2, d=d, dh=dh, dtype=dtype,
                            opt=opt, seed=base.seed + 9000 + d + dh).with_tokens(n, chunk=256)
    inp = li.make_inputs(w)
    got = run_gpu(w, inp)
    want = O.run_workload(w, inp)
    errs = compare(w, got, want, "corner")
    assert max(errs.values()) < TOL[w.dtype], errs
    dW = compare_change(w, initial_weights(w, inp), got[1:], want[1:], exact_gradient=False, test="corner")
    assert max(dW.values()) < dw_tol(w, False), dW


@pytest.mark.parametrize("num", [4, 10, 3])
def test_set_call_with_no_update_tokens_reads_the_initial_memory(num):
    # lact_sequence in the set order with n_kv = 0: the (empty) update leaves
    # W bit for bit, and the queries read the initial fast weights
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(0, n_q=300, chunk=1, seed=li.WORKLOADS[num].seed + 8200)
    w = dataclasses.replace(w, order="set")
    inp = li.make_inputs(w)
    layer = _layer(w, inp, max_chunk=1)
    before = [None if x is None else x.clone() for x in layer.weights()]
    q = to_device(inp.q)
    z = torch.zeros(16, device="cuda")
    o = torch.empty_like(q)
    L.lact_sequence(layer.handle, L.LACT_SET_UPDATE_THEN_APPLY, q, w.n_q, z, z, z, 0, 1, o)
    after = layer.weights()
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    for x, y in zip(before, after):
        assert (x is None and y is None) or torch.equal(x, y)
    got = to_host_f64(o)
    mats = (inp.W1,) if w.memory == "linear" else (inp.W1, inp.W2, inp.W3)
    for b in range(w.B):
        for h in range(w.H):
            want = O.memory_apply(tuple(x[h].astype(np.float64) for x in mats), li.as_f64(inp.q[b, h]))
            err = np.linalg.norm(got[b, h] - want) / np.linalg.norm(want)
            assert err < TOL[w.dtype], (b, h, err)


def test_set_call_with_no_queries_still_updates():
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[4].with_tokens(1000 + 3, n_q=0, seed=li.WORKLOADS[4].seed + 8300)
    inp = li.make_inputs(w)
    layer = _layer(w, inp, max_chunk=w.n_kv)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    z = torch.zeros(16, device="cuda")
    L.lact_sequence(layer.handle, L.LACT_SET_UPDATE_THEN_APPLY, z, 0, k, v, e, w.n_kv, w.n_kv, z)
    got = [to_host_f64(x) for x in layer.weights()]
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    want = O.run_workload(w, inp)
    errs = compare(w, (None,) + tuple(got), (None,) + tuple(want[1:]), "no_queries")
    assert max(errs.values()) < TOL[w.dtype], errs


def test_two_states_on_two_streams_run_independently():
    # two layers, each on its own stream, launched interleaved: the results
    # equal those of the same calls made one after the other
    import torch
    from chunk_test_step_b300 import lact as L
    ws = [li.WORKLOADS[8].with_tokens(4096 + 11, seed=li.WORKLOADS[8].seed + 8400),
          li.WORKLOADS[2].with_tokens(2048 + 5, seed=li.WORKLOADS[2].seed + 8400)]
    inps = [li.make_inputs(w) for w in ws]

    def run(concurrent):
        layers = [_layer(w, inp) for w, inp in zip(ws, inps)]
        ios = [tuple(to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta)) for inp in inps]
        outs = [torch.empty_like(io[0]) for io in ios]
        streams = [torch.cuda.Stream(), torch.cuda.Stream()] if concurrent else [torch.cuda.current_stream()] * 2
        torch.cuda.synchronize()
        for i, (w, layer, (q, k, v, e), o, s) in enumerate(zip(ws, layers, ios, outs, streams)):
            L.lact_sequence(layer.handle, L.LACT_CAUSAL_APPLY_THEN_UPDATE, q, w.n_q, k, v, e, w.n_kv, w.chunk, o, s)
        torch.cuda.synchronize()
        res = [[o.clone()] + [x.clone() for x in layer.weights() if x is not None] for layer, o in zip(layers, outs)]
        torch.cuda.synchronize()
        for layer in layers:
            assert L.lact_sync_status(layer.handle) == L.LACT_OK
            layer.close()
        return res

    seq, conc = run(False), run(True)
    for a, b in zip(seq, conc):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("mat", [0, 1])
def test_nonfinite_weight_sets_status_in_the_fused_muon_step(mat):
    # a NaN in W1 (tall) or W2 (wide) on the bf16 Muon layer: Newton-Schulz's
    # own update finds a non-finite row norm and sets the sticky status
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[4].with_tokens(256, seed=li.WORKLOADS[4].seed + 8500)
    inp = li.make_inputs(w)
    layer = _layer(w, inp, max_chunk=w.n_kv)
    Ws = list(layer.weights())
    Ws[mat][0, 0, 3, 5] = float("nan")
    L.lact_set_weights(layer.handle, *Ws)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    L.lact_chunk_update(layer.handle, k, v, e, w.n_kv)
    assert L.lact_sync_status(layer.handle) == L.LACT_ERR_NONFINITE
