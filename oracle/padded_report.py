"""What padding every expert batch to one capacity would cost on a workload.

TEST INFRASTRUCTURE (fp64 CPU oracle): a command-line report, run by hand; the
product path never imports it.

    python -m oracle.padded_report skew_e128 [--seed 0] [--factor 1.25]

OLMo-core 3 tutorial, section "另外两处税：主机同步与 padding": the grouped GEMM
runs each expert on its exact routed rows instead of padding every expert
batch to a common capacity.  For the workload's routing this prints, as one
JSON line, the capacity C = ceil(factor * T * k / E), the spread of the
expert loads, how many routed rows a capacity-C layer drops (first C rows of
each expert in token order are kept), the rows that layer multiplies (E * C)
against the T * k rows of the unpadded one, and the relative L2 distance of
its output from the unpadded layer's output (both fp64, from the same bf16
inputs and the same fp32 router logits).
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import layer as ol          # noqa: E402
from oracle import padded as pd         # noqa: E402
from token_dispatch_grouped_router_gb300 import workloads as wl   # noqa: E402


def report(key: str, seed: int = 0, factor: float = 1.25) -> dict:
    w = wl.get_workload(key)
    inp = wl.generate(w, seed=seed, with_backward=False)
    t0 = time.perf_counter()
    fwd = ol.layer_forward(inp, w.k, w.E)
    counts = np.asarray(fwd["counts"], np.int64)
    C = pd.capacity(w.T, w.k, w.E, factor)
    p = pd.padded_forward(inp["x"], fwd["idx"], fwd["g"], inp["W1"], inp["W3"], inp["W2"], w.E, C)
    diff = p["out"] - fwd["out"]
    rel_l2 = float(np.linalg.norm(diff) / np.linalg.norm(fwd["out"]))
    tokens_hit = int((~p["kept"]).any(axis=1).sum())
    return {
        "workload": w.name, "seed": seed, "capacity_factor": factor, "capacity": C,
        "routed_rows": int(w.R), "mean_load": w.R / w.E, "max_load": int(counts.max()),
        "max_over_mean": float(counts.max() / (w.R / w.E)),
        "empty_experts": int((counts == 0).sum()),
        "experts_over_capacity": int((counts > C).sum()),
        "dropped_rows": p["dropped"], "dropped_fraction": p["dropped_fraction"],
        "tokens_with_a_dropped_expert": tokens_hit,
        "padded_rows": p["padded_rows"], "unpadded_rows": p["unpadded_rows"],
        "padded_over_unpadded_gemm_flops": p["padded_rows"] / p["unpadded_rows"],
        "padded_rows_that_are_zero": int(w.E * C - (w.R - p["dropped"])),
        "rel_l2_padded_vs_unpadded_out": rel_l2,
        "oracle_seconds": time.perf_counter() - t0,
    }


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("key", nargs="?", default="skew_e128")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--factor", type=float, default=1.25)
    a = ap.parse_args()
    print(json.dumps(report(a.key, a.seed, a.factor)))


if __name__ == "__main__":
    main()
