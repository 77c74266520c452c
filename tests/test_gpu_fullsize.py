"""Full-size parity: every workload at its own size, in the launch
configuration bench.py times (one lact_sequence call, max_chunk = chunk; for
the bf16 workloads the call captured as a CUDA graph and replayed, as the
bench times it).

The tiny fp32 workloads are compared with the oracle element by element.
For the bf16 workloads the oracle cannot run inside a test (the
million-token layer is ~6.6e12 fp64 FLOP), so tests/golden/ holds a fixed
random sample of rows of o and of the final W1, W2, W3 per (b, h), written
by tests/golden/make_golden.py from the oracle alone; the sampled rows must
match within the bf16 budget (relative L2 error 2e-2 per tensor per (b, h)).
A property that holds at any size is checked on every row: each row of the
final weights keeps the L2 norm of the initial weights (renorm to the
pre-update norm, which itself equals the initial norm by induction).
"""
import json
import os

import numpy as np
import pytest

import lact_inputs as li
from oracle import lact_oracle as O
from tests.harness import TOL, compare, compare_change, config_for, dw_tol, initial_weights, record, rel_l2, run_gpu, to_device

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("num", [1, 3, 6, 9])
def test_tiny_workloads_full_size(num):
    w = li.WORKLOADS[num]
    inp = li.make_inputs(w)
    got, want = run_gpu(w, inp), O.run_workload(w, inp)
    errs = compare(w, got, want, "fullsize")
    assert max(errs.values()) < TOL[w.dtype], errs
    dW = compare_change(w, initial_weights(w, inp), got[1:], want[1:], exact_gradient=False, test="fullsize")
    assert max(dW.values()) < dw_tol(w, False), dW


@pytest.mark.parametrize("num", [2, 4, 5, 7, 8, 10])
def test_bf16_workloads_full_size_sampled(num):
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num]
    doc = json.load(open(os.path.join(GOLDEN, f"fullsize_{w.name}.json")))
    assert doc["seed"] == w.seed
    inp = li.make_inputs(w)
    layer = L.LactLayer(config_for(w), to_device(inp.W1), to_device(inp.W2), to_device(inp.W3))
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    o = torch.empty_like(q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lact_sequence(layer.handle, order, q, w.n_q, k, v, e, w.n_kv, w.chunk, o, s)
    torch.cuda.synchronize()
    g.replay()              # the one step, from the initial weights
    W = layer.weights()
    torch.cuda.synchronize()
    assert L.lact_sync_status(layer.handle) == L.LACT_OK
    W0 = (inp.W1, inp.W2, inp.W3)
    worst = {}
    tol_dw = dw_tol(w, exact_gradient=False)
    for head in doc["heads"]:
        b, h, rows = head["b"], head["h"], head["rows"]
        got_o = o[b, h, rows["o"]].double().cpu().numpy()
        err = rel_l2(got_o, np.array(head["o"]))
        worst["o"] = max(worst.get("o", 0.0), err)
        assert err < TOL["bf16"], ("o", b, h, err)
        for m, name in enumerate(("W1", "W2", "W3")):
            if W[m] is None:
                continue
            got = W[m][b, h, rows[name]].double().cpu().numpy()
            want = np.array(head[name])
            err = rel_l2(got, want)
            worst[name] = max(worst.get(name, 0.0), err)
            assert err < TOL["bf16"], (name, b, h, err)
            # the change of the sampled rows over the call (initial rows are
            # the generator's, the final ones the oracle's)
            w0 = W0[m][h, rows[name]].astype(np.float64)
            chg = rel_l2(got - w0, want - w0)
            worst["d" + name] = max(worst.get("d" + name, 0.0), chg)
            assert chg < tol_dw, ("d" + name, b, h, chg)
    for name, err in worst.items():
        record("fullsize_sampled", w, name, err, tol_dw if name.startswith("d") else TOL["bf16"],
               **({"kind": "change"} if name.startswith("d") else {}))
    # every row keeps its initial norm
    for m in range(3):
        if W[m] is None:
            continue
        n_got = torch.linalg.vector_norm(W[m].double(), dim=-1).cpu().numpy()
        n_0 = np.linalg.norm(W0[m].astype(np.float64), axis=-1)
        np.testing.assert_allclose(n_got, np.broadcast_to(n_0, n_got.shape), rtol=1e-5)
    layer.close()
