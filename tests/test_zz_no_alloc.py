"""The allocation-free chunk gradient (lact_chunk_gradient_noalloc).

It serves callers that cannot allocate device memory, so it keeps its
split-K partial sums in static device memory inside liblact instead of a
caller-provided workspace. This file is collected last on purpose: if it
fails, every other test has already run.

Checks, through the C ABI: two calls in a row match the workspace-based
lact_chunk_gradient and the fp64 oracle within the bf16 parity budget (max
relative L2 error 2e-2 per matrix per (b, h)); the device's free memory is
the same before and after the second call (the first one may load the
library's device code, which allocates); a problem too large for the static
scratch, and the linear memory, are refused before anything runs.
"""
import numpy as np
import pytest

import lact_inputs as li
from oracle import lact_oracle as O
from tests.harness import TOL, config_for, record, rel_l2, to_device, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("num,n", [(4, 3000 + 41), (2, 1024 + 7)])
def test_noalloc_gradient_matches_workspace_gradient_twice(num, n):
    import torch
    from chunk_test_step_b300 import lact as L
    w = li.WORKLOADS[num].with_tokens(n, seed=li.WORKLOADS[num].seed + 4000)
    inp = li.make_inputs(w)
    cfg = config_for(w, max_chunk=n)
    layer = L.LactLayer(cfg, to_device(inp.W1), to_device(inp.W2), to_device(inp.W3))
    k, v, e = to_device(inp.k), to_device(inp.v), to_device(inp.eta)
    shapes = ((w.dh, w.d), (w.d, w.dh), (w.dh, w.d))
    ref = [torch.empty(w.B, w.H, *s, device="cuda") for s in shapes]
    L.lact_chunk_gradient(layer.handle, k, v, e, n, *ref)
    W = layer.weights()                      # [B, H, ...] fp32, the state's weights
    outs = [[torch.full((w.B, w.H) + s, float("nan"), device="cuda") for s in shapes] for _ in range(2)]
    torch.cuda.synchronize()
    L.lact_chunk_gradient_noalloc(cfg, *W, k, v, e, n, *outs[0])   # may load the device code
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    L.lact_chunk_gradient_noalloc(cfg, *W, k, v, e, n, *outs[1])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    ref = [to_host_f64(x) for x in ref]
    want = [O.chunk_gradient(inp.W1[h].astype(np.float64), inp.W2[h].astype(np.float64),
                             inp.W3[h].astype(np.float64), li.as_f64(inp.k[b, h]), li.as_f64(inp.v[b, h]),
                             inp.eta[b, h].astype(np.float64)) for b in range(w.B) for h in range(w.H)]
    for g in outs:
        got = [to_host_f64(x) for x in g]
        for m in range(3):
            for b in range(w.B):
                for h in range(w.H):
                    err = rel_l2(got[m][b, h], ref[m][b, h])
                    assert err < TOL["bf16"], (m, b, h, err)
                    err = record("noalloc_gradient", w, "gW%d" % (m + 1),
                                 rel_l2(got[m][b, h], want[b * w.H + h][m]), TOL["bf16"], b=b, h=h)
                    assert err < TOL["bf16"], ("oracle", m, b, h, err)
    for m in range(3):   # same work, same order: the two calls agree exactly
        assert torch.equal(outs[0][m], outs[1][m])
    layer.close()


def test_noalloc_gradient_rejects_problems_beyond_its_scratch():
    import torch
    from chunk_test_step_b300 import lact as L
    # one split slot = 12 * B*H*d*dh bytes = 36 MiB > 32 MiB
    cfg = L.make_config(2, 8, 256, 768, "bf16", "gd", max_chunk=128)
    z = torch.zeros(16, device="cuda")
    with pytest.raises(L.LactError) as ex:
        L.lact_chunk_gradient_noalloc(cfg, z, z, z, z, z, z, 0, z, z, z)
    assert ex.value.status == L.LACT_ERR_UNSUPPORTED


def test_noalloc_gradient_rejects_the_linear_memory():
    import torch
    from chunk_test_step_b300 import lact as L
    cfg = L.make_config(1, 2, 128, 128, "bf16", "gd", max_chunk=128, memory="linear")
    z = torch.zeros(16, device="cuda")
    with pytest.raises(L.LactError) as ex:
        L.lact_chunk_gradient_noalloc(cfg, z, z, z, z, z, z, 0, z, z, z)
    assert ex.value.status == L.LACT_ERR_UNSUPPORTED
