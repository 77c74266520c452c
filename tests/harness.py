"""Shared helpers of the parity tests: run a workload through the C ABI (via
the Python binding) and through the oracle, and compare them."""
from __future__ import annotations

import numpy as np

import lact_inputs as li

# Parity budgets (max relative L2 error per tensor per (b, h)): 1e-4 for the
# fp32 workloads, 2e-2 for the bf16-input workloads.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def dw_tol(w: li.Workload, exact_gradient: bool) -> float:
    """Budget of the weight CHANGE dW = W_after - W_before, relative to |dW_ref|.

    The final-weight budget above is relative to |W|, and one update moves W
    by 1-3 % of its norm, so that budget alone cannot see a wrong update. The
    change itself is compared against these bounds, derived from the
    arithmetic (an emulation of the bf16 tensor-core path in numpy: bf16
    operands at the rounding points the kernels use, fp32 accumulation):

    * fp32 io computes in fp64 inside: 1e-4, the fp32 budget.
    * bf16 io, gradient descent or momentum: the change is the gradient, whose
      bf16 operands (u', dh1, dh3 rounded) put it 2.9e-3 from the fp64 one:
      2e-2, the bf16 budget.
    * bf16 io, Muon from a gradient given exactly (lact_apply_gradient): only
      the accumulation order differs from the oracle's (fp32 vs fp64), which
      flips a few bf16 roundings of X, A, B. The quintic map's slope (3.4 near
      0, |p'| up to 1.6 in its band) amplifies each flip: emulated drift
      <= 1.2e-6 after 1 step, 2.2e-5 after 2, 1.3e-3 after 3, 1.4e-2 after 5.
      Budgets 1e-3 (<= 2 steps), 1e-2 (3 steps), 2e-2 (5 steps).
    * bf16 io, Muon from the tensor-core gradient (whole layer calls): the
      gradient's own 2.9e-3 passes through that amplification: emulated
      2.9e-3 after <= 2 steps, 2.1e-2 - 2.4e-2 after 5 (the four bf16 Muon
      layers, every matrix). Budgets 2e-2 (<= 2 steps) and 5e-2 (5 steps).
    """
    if w.dtype == "f32":
        return 1e-4
    if w.opt != "muon":
        return 2e-2
    if exact_gradient:
        return 1e-3 if w.ns_steps <= 2 else (1e-2 if w.ns_steps <= 3 else 2e-2)
    return 2e-2 if w.ns_steps <= 2 else 5e-2


# Measured parity: every comparison the tests make is appended here, and the
# session writes the list as JSON to the path in LACT_PARITY_LOG (if set).
RECORDS: list = []


def record(test: str, w: li.Workload, tensor: str, err: float, tol: float, **extra) -> float:
    RECORDS.append(dict(test=test, workload=w.number, name=w.name, n_kv=w.n_kv, n_q=w.n_q,
                        opt=w.opt, ns_steps=w.ns_steps, tensor=tensor, err=float(err), tol=float(tol), **extra))
    return err


def rel_l2(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    num = np.linalg.norm(got - want)
    return float(num / den) if den > 0 else float(num)


def max_rel_l2_per_head(got, want) -> float:
    """got, want: [B, H, ...]; max over (b, h) of the rel-L2 of each slice."""
    B, H = want.shape[:2]
    return max(rel_l2(got[b, h], want[b, h]) for b in range(B) for h in range(H))


def to_device(a: np.ndarray, device="cuda"):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_host_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def config_for(w: li.Workload, max_chunk: int | None = None):
    from chunk_test_step_b300 import lact as L
    return L.make_config(w.B, w.H, w.d, w.dh, w.dtype, w.opt,
                         max_chunk=max_chunk or max(w.chunk, 1), ns_steps=w.ns_steps,
                         ns_a=w.ns_a, ns_b=w.ns_b, ns_c=w.ns_c, muon_lr=w.muon_lr, momentum=w.momentum,
                         memory=w.memory)


def run_gpu(w: li.Workload, inp: li.Inputs):
    """lact_sequence on the GPU; returns (o, W1, W2, W3) as fp64 numpy arrays."""
    import torch
    from chunk_test_step_b300 import lact as L
    layer = L.LactLayer(config_for(w), to_device(inp.W1), to_device(inp.W2), to_device(inp.W3))
    q, k, v, e = (to_device(x) for x in (inp.q, inp.k, inp.v, inp.eta))
    order = L.LACT_CAUSAL_APPLY_THEN_UPDATE if w.order == "causal" else L.LACT_SET_UPDATE_THEN_APPLY
    o = layer.sequence(order, q, k, v, e, w.chunk)
    W1, W2, W3 = layer.weights()
    torch.cuda.synchronize()
    st = L.lact_sync_status(layer.handle)
    assert st == L.LACT_OK, L.lact_status_str(st)
    out = tuple(None if x is None else to_host_f64(x) for x in (o, W1, W2, W3))
    layer.close()
    return out


def compare(w: li.Workload, got, want, test: str = "") -> dict:
    names = ("o", "W1", "W2", "W3")
    errs = {n: max_rel_l2_per_head(g, r) for n, g, r in zip(names, got, want) if r is not None}
    for n, e in errs.items():
        record(test, w, n, e, TOL[w.dtype])
    return errs


def initial_weights(w: li.Workload, inp: li.Inputs):
    """The initial fast weights per (b, h) as fp64 [B, H, ...] (head h's for every b)."""
    return tuple(None if x is None else np.broadcast_to(x.astype(np.float64)[None], (w.B,) + x.shape)
                 for x in (inp.W1, inp.W2, inp.W3))


def compare_change(w: li.Workload, W0, got, want, exact_gradient: bool, test: str = "") -> dict:
    """Max over (b, h) of the rel-L2 error of the weight change got - W0
    against want - W0, per matrix; each is recorded against dw_tol."""
    errs = {}
    tol = dw_tol(w, exact_gradient)
    for n, w0, g, r in zip(("dW1", "dW2", "dW3"), W0, got, want):
        if r is None:
            continue
        errs[n] = max_rel_l2_per_head(g - w0, r - w0)
        record(test, w, n, errs[n], tol, kind="change")
    return errs
