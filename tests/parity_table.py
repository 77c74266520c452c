"""Summarise the parity log the GPU tests write (LACT_PARITY_LOG=file).

    LACT_PARITY_LOG=parity.json python -m pytest tests -m gpu
    python tests/parity_table.py parity.json

Prints, per test and workload, the worst relative L2 error of each compared
tensor (o, W1..W3, the gradient gW*, and the weight change dW*) against its
budget, as markdown. It reads only the log.
"""
import json
import sys
from collections import defaultdict


def main(path: str) -> None:
    worst, tol = defaultdict(float), {}
    for r in json.load(open(path)):
        key = (r["test"], r["name"], r["ns_steps"] if r["opt"] == "muon" else None, r["tensor"])
        worst[key] = max(worst[key], r["err"])
        tol[key] = r["tol"]
    print("| test | workload | NS steps | tensor | worst rel-L2 | budget | headroom |")
    print("|---|---|---|---|---:|---:|---:|")
    for key in sorted(worst, key=lambda k: (k[0], k[1], k[2] or 0, k[3])):
        t, name, ns, tensor = key
        e = worst[key]
        print(f"| {t} | {name} | {ns if ns is not None else ''} | {tensor} | {e:.2e} | {tol[key]:.0e} | "
              f"{tol[key] / e if e > 0 else float('inf'):.0f}x |")


if __name__ == "__main__":
    main(sys.argv[1] if len(sys.argv) > 1 else "parity.json")
