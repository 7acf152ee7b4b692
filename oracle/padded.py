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

from .layer import _f64, _sigmoid, router_topk_backward, silu, route_map

__all__ = ["capacity", "capacity_route_map", "padded_forward", "padded_backward"]


def capacity(T: int, k: int, E: int, factor: float = 1.25) -> int:
    return int(math.ceil(factor * T * k / E))


def capacity_route_map(idx: np.ndarray, E: int, C: int):
    """Route map of the padded layer: expert e owns rows [e*C, (e+1)*C).

    Returns counts[E] (rows kept, min(routed, C)), offsets[E+1] (e*C),
    row_of_slot[T*k] (e*C + the slot's rank among the slots routed to e in
    slot order when that rank is below C, else -1 for a dropped slot),
    slot_of_row[E*C] (the slot a row holds, -1 for a zero row) and routed[E]
    (rows routed before the cut), all int32.
    """
    idx = np.asarray(idx, np.int64)
    flat = idx.reshape(-1)
    routed = np.zeros(E, np.int64)
    row_of_slot = np.full(flat.size, -1, np.int64)
    slot_of_row = np.full(E * C, -1, np.int64)
    for s, e in enumerate(flat):                 # slots in order: rank = earlier slots of e
        rank = routed[e]
        routed[e] += 1
        if rank < C:
            row_of_slot[s] = e * C + rank
            slot_of_row[e * C + rank] = s
    counts = np.minimum(routed, C)
    offsets = np.arange(E + 1, dtype=np.int64) * C
    i32 = lambda a: a.astype(np.int32)  # noqa: E731
    return i32(counts), i32(offsets), i32(row_of_slot), i32(slot_of_row), i32(routed)


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


def padded_backward(x, idx, g, W1, W3, W2, dOut, E: int, C: int, W_r=None) -> Dict:
    """Backward of padded_forward for the upstream gradient dOut (fp64).

    The padded layer computes out[t] = sum over the KEPT slots (t, j) of
    g[t,j] * FFN_e(x[t]), each expert on a batch of exactly C rows (its first
    C routed rows in token order, then zero rows).  Its gradients:
      dg[t,j]  = <dOut[t], FFN_e(x[t])> for a kept slot, 0 for a dropped one;
      per expert, with dY_b[r] = g[t,j] dOut[t] on the kept rows and 0 on the
      zero rows, the SwiGLU backward of the batch (dA = dY_b W2^T,
      dH1 = dA H3 silu'(H1), dH3 = dA silu(H1), dX_b = dH1 W1^T + dH3 W3^T,
      dW2 = A^T dY_b, dW1 = X_b^T dH1, dW3 = X_b^T dH3);
      dX[t] = sum over its kept slots of the batch row's dX_b;
      dz = the renormalised top-k softmax backward of dg (a dropped slot's
      gate still enters the softmax normaliser, so its logit gets gradient);
      for a learned router (W_r given) dX += dz W_r^T, dW_r = x^T dz,
      db = sum_t dz.
    """
    x = _f64(x); g = _f64(g); dOut = _f64(dOut)
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    d = x.shape[1]
    h = np.asarray(W1).shape[2]
    counts, offsets, row_of_slot, slot_of_row = route_map(idx, E)
    dX = np.zeros((T, d))
    dg = np.zeros((T, k))
    dW1 = np.zeros((E, d, h)); dW3 = np.zeros((E, d, h)); dW2 = np.zeros((E, h, d))
    for e in range(E):
        slots = slot_of_row[offsets[e]:offsets[e + 1]].astype(np.int64)
        keep = slots[:C]
        batch = np.zeros((C, d))
        batch[:keep.size] = x[keep // k]
        dYb = np.zeros((C, d))
        for r, s in enumerate(keep):
            dYb[r] = g[s // k, s % k] * dOut[s // k]
        H1 = batch @ _f64(W1[e]); H3 = batch @ _f64(W3[e])
        A = silu(H1) * H3
        Y = A @ _f64(W2[e])
        dA = dYb @ _f64(W2[e]).T
        sg = _sigmoid(H1)
        dH1 = dA * H3 * sg * (1.0 + H1 * (1.0 - sg))
        dH3 = dA * H1 * sg
        dXb = dH1 @ _f64(W1[e]).T + dH3 @ _f64(W3[e]).T
        dW2[e] = A.T @ dYb
        dW1[e] = batch.T @ dH1
        dW3[e] = batch.T @ dH3
        for r, s in enumerate(keep):
            dg[s // k, s % k] = float(dOut[s // k] @ Y[r])
            dX[s // k] += dXb[r]
    dz = router_topk_backward(g, dg, idx, E)
    res = {"dX_expert": dX.copy(), "dg": dg, "dW1": dW1, "dW3": dW3, "dW2": dW2, "dz": dz}
    if W_r is not None:
        Wr = _f64(W_r)
        dX += dz @ Wr.T
        res.update(dW_r=x.T @ dz, db=dz.sum(axis=0))
    res["dX"] = dX
    return res
