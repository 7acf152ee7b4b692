"""Padded-to-capacity expert batches: the alternative the method removes.

TEST INFRASTRUCTURE (fp64 CPU oracle), imported only by tests and the
benchmark's CPU-baseline leg.

OLMo-core 3 tutorial, section "另外两处税：主机同步与 padding": the device-side
grouped GEMM runs each expert on its exact row count instead of padding every
expert batch to one common capacity; the speed-read summary of the report
("GPU-resident metadata removes recurring host waits") says it measures where
that beats the padded alternative.  The pages give no capacity formula.  The
reading used here: capacity C = ceil(1.25 * T * k / E); every expert keeps its
first C routed rows in token order and drops the rest; a dropped slot
contributes zero to its token's output and the other gates are not
renormalised.
"""
from __future__ import annotations

import math
from typing import Dict

import numpy as np

from .layer import _f64, silu, route_map

__all__ = ["capacity", "padded_forward"]


def capacity(T: int, k: int, E: int, factor: float = 1.25) -> int:
    return int(math.ceil(factor * T * k / E))


def padded_forward(x, idx, g, W1, W3, W2, E: int, C: int) -> Dict:
    """Forward with per-expert batches of exactly C rows (zero rows pad short
    experts; rows past C are dropped).

    Returns the output, the kept mask per slot, dropped count and fraction,
    and the row counts the padded and unpadded GEMMs multiply.
    """
    x = _f64(x); g = _f64(g)
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    counts, offsets, row_of_slot, slot_of_row = route_map(idx, E)
    kept = np.zeros(T * k, bool)
    out = np.zeros((T, x.shape[1]))
    for e in range(E):
        # the expert's slots in token order (its route-map segment)
        slots = slot_of_row[offsets[e]:offsets[e + 1]].astype(np.int64)
        keep = slots[:C]
        kept[keep] = True
        batch = np.zeros((C, x.shape[1]))          # padded expert batch
        batch[:keep.size] = x[keep // k]
        Y = (silu(batch @ _f64(W1[e])) * (batch @ _f64(W3[e]))) @ _f64(W2[e])
        for r, s in enumerate(keep):
            out[s // k] += g[s // k, s % k] * Y[r]
    dropped = int((~kept).sum())
    return {"out": out, "kept": kept.reshape(T, k), "dropped": dropped,
            "dropped_fraction": dropped / float(T * k),
            "padded_rows": E * C, "unpadded_rows": T * k}
