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


@pytest.mark.parametrize("num", [4, 1])
def test_zero_weight_row_stays_zero(num):
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(1000 + 37, seed=li.WORKLOADS[num].seed + 8000)
    inp = li.make_inputs(w)
    W1 = inp.W1.copy()
    W1[:, 5, :] = 0.0                       # hidden unit 5 of every head: W1 row of zeros
    inp = dataclasses.replace(inp, W1=W1)
    n = w.n_kv
    layer = _layer(w, inp, max_chunk=n)
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    L.lact_chunk_update(layer.handle, k, v, e, n)
    got = [to_host_f64(x) for x in layer.weights()]
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    assert np.all(got[0][:, :, 5, :] == 0.0)
    for b in range(w.B):
        for h in range(w.H):
            Wf = O.chunk_update(tuple(x[h].astype(np.float64) for x in (inp.W1, inp.W2, inp.W3)),
                                li.as_f64(inp.k[b, h]), li.as_f64(inp.v[b, h]), inp.eta[b, h].astype(np.float64),
                                w.opt, lr=w.muon_lr, ns_steps=w.ns_steps)
            assert np.all(Wf[0][5] == 0.0)
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
