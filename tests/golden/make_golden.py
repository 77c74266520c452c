"""Write the sampled full-size expected values of tests/test_gpu_fullsize.py.

Runs the fp64 oracle (oracle/) on the full-size bf16 workloads (the
language-model causal layers with GD and with momentum, the 3B-shaped
causal layer, the 48-view image-set layer, the million-token set layer and
the image-set layer with the linear memory)
with the seeded inputs of
lact_inputs, and stores,
per (b, h), a fixed random sample of rows of the output o and of the final
fast weights W1, W2, W3. Nothing here comes from the CUDA path.

    python tests/golden/make_golden.py [workload numbers, default 2 4 5 7 8 10]

Takes minutes (the million-token layer is ~6.6e12 fp64 FLOP).
"""
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import lact_inputs as li  # noqa: E402
from oracle import lact_oracle as O  # noqa: E402

O_ROWS, W_ROWS = 8, 4


def sample_indices(w: li.Workload):
    """Fixed per-workload sample of row indices (same in the test)."""
    g = np.random.default_rng(w.seed + 777)
    out = []
    for _ in range(w.B * w.H):
        out.append({
            "o": sorted(g.choice(w.n_q, size=O_ROWS, replace=False).tolist()),
            "W1": sorted(g.choice(w.dh, size=W_ROWS, replace=False).tolist()),
            "W2": sorted(g.choice(w.d, size=W_ROWS, replace=False).tolist()),
            "W3": sorted(g.choice(w.dh, size=W_ROWS, replace=False).tolist()),
            # (the linear memory has W1 only, [d, d]: its rows come from the W1 draw)
        })
    return out


def main(nums):
    for num in nums:
        w = li.WORKLOADS[num]
        t0 = time.time()
        inp = li.make_inputs(w)
        Of, W1, W2, W3 = O.run_workload(w, inp, token_slice=65536)
        idx = sample_indices(w)
        heads = []
        for bh, sel in enumerate(idx):
            b, h = divmod(bh, w.H)
            heads.append({
                "b": b, "h": h, "rows": sel,
                "o": [[float(f"{x:.8e}") for x in Of[b, h, i]] for i in sel["o"]],
                "W1": [[float(f"{x:.8e}") for x in W1[b, h, i]] for i in sel["W1"]],
                "W2": [] if W2 is None else [[float(f"{x:.8e}") for x in W2[b, h, i]] for i in sel["W2"]],
                "W3": [] if W3 is None else [[float(f"{x:.8e}") for x in W3[b, h, i]] for i in sel["W3"]],
            })
        doc = {"workload": w.name, "number": num, "seed": w.seed,
               "written_by": "tests/golden/make_golden.py (fp64 oracle)", "heads": heads}
        path = os.path.join(HERE, f"fullsize_{w.name}.json")
        with open(path, "w") as f:
            json.dump(doc, f, separators=(",", ":"))
        print(f"{w.name}: {time.time() - t0:.1f} s -> {path}", flush=True)


if __name__ == "__main__":
    main([int(x) for x in sys.argv[1:]] or [2, 4, 5, 7, 8, 10])
