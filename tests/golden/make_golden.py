"""Writes tests/golden/oracle_small.json: the oracle's forward on one fixed tiny input.

A regression fixture for the oracle itself (it calls only ``oracle`` and the
seeded generator in ``workloads``).  Inputs are multiples of 1/64 so that the
text form is exact.  Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import make_cu_seqlens, make_selection  # noqa: E402


def main():
    seqlens, h_k, g, d, block, topk, scale = [10, 14], 1, 2, 4, 4, 3, 0.5
    n = sum(seqlens)
    rng = np.random.default_rng(2024)
    sel = make_selection(seqlens, h_k, block, topk, "uniform", rng)
    q = np.round(rng.standard_normal((n, h_k * g, d)) * 64) / 64
    k = np.round(rng.standard_normal((n, h_k, d)) * 64) / 64
    v = np.round(rng.standard_normal((n, h_k, d)) * 64) / 64
    cu = make_cu_seqlens(seqlens)
    out, lse = oracle.fwd(cu, block, sel, q, k, v, scale)
    gold = {
        "about": "oracle forward on a fixed tiny packed batch (regression fixture); "
                 "written by tests/golden/make_golden.py",
        "inputs": {"cu_seqlens": cu.tolist(), "block": block, "scale": scale,
                   "sel_idx": sel.tolist(), "q": q.tolist(), "k": k.tolist(), "v": v.tolist()},
        "out": out.tolist(), "lse": lse.tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as f:
        json.dump(gold, f, indent=None, separators=(",", ":"))
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
