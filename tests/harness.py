"""Shared helpers of the parity tests: run a workload through the C ABI (via
the Python binding) and through the oracle, and compare them."""
from __future__ import annotations

import numpy as np

import lact_inputs as li

# Parity budgets (max relative L2 error per tensor per (b, h)): 1e-4 for the
# fp32 workloads, 2e-2 for the bf16-input workloads.
TOL = {"f32": 1e-4, "bf16": 2e-2}


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


def compare(w: li.Workload, got, want) -> dict:
    names = ("o", "W1", "W2", "W3")
    return {n: max_rel_l2_per_head(g, r) for n, g, r in zip(names, got, want) if r is not None}
