"""fp64 CPU oracle of the single-GPU MoE expert layer (forward and backward).

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The product path never
calls it, and it shares no code, tables or helpers with the CUDA library.

What the layer computes is the plain, unfused MoE feed-forward layer; the
pages' method reaches exactly this result with less data movement:

* OLMo-core 3 tutorial (bloombook.cn), section "rowwise EP：用 NVSHMEM 一端直写":
  each routed token row is written straight into its expert's input buffer by
  looking up the routing table, and combine brings the expert outputs back.
* same page, section "另外两处税：主机同步与 padding": routing counts, rows per
  expert and the per-expert permutation form a device-resident route map, and
  the grouped GEMM runs each expert on exactly its routed rows, unpadded.
* "Ai2 Olmo-core 3: The Secret Behind 2.7x MoE Training Throughput", section
  "The Capacity Tax": each token activates a few experts (e.g. 4 of 128)
  chosen by a routing function.

The pages do not define the routing function, the expert network or the
intermediate precisions.  The readings used here (the benchmark
specification's) are:

* router: softmax over the E logits, then top-k; selection is done on the fp32
  logits (softmax is monotone), ties go to the lower expert id, and the k gates
  are the softmax renormalised over the selected logits;
* slot order within a token: descending logit;
* rows of one expert's segment: ascending flattened slot t*k+j (stable);
* expert FFN: SwiGLU, Y = (silu(X W1) * (X W3)) W2, no biases;
* everything here in fp64 with no intermediate rounding.

Every array argument may be fp64 already; bf16 inputs arrive as uint16 bit
patterns and are decoded by ``decode_bf16``.
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

__all__ = [
    "decode_bf16", "router_logits", "topk", "softmax_gates", "topk_gates",
    "route_map", "dispatch", "silu", "expert_ffn_forward", "combine",
    "combine_backward", "expert_ffn_backward", "unpermute_sum",
    "router_topk_backward", "router_logits_backward", "layer_forward",
    "layer_backward",
]


# ---------------------------------------------------------------------------
# storage decode
# ---------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    b = np.asarray(bits)
    if b.dtype != np.uint16:
        raise TypeError("bf16 tensors are passed as uint16 bit patterns")
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return decode_bf16(a)
    return a.astype(np.float64)


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------

def router_logits(x, W_r, b=None, out_dtype=np.float32) -> np.ndarray:
    """z = x W_r (+ b): computed in fp64 from the stored inputs, returned as fp32
    (``out_dtype=np.float64`` keeps fp64, for finite-difference checks).

    The router stays in high precision, as the DeepSeek-V3 recipe keeps gating
    out of FP8 (OLMo-core 3 tutorial, section "一个低精度格式，同时压三个地方",
    DeepSeek-V3 paragraph).  The fp32 result is what both top-k paths consume.
    """
    z = _f64(x) @ _f64(W_r)
    if b is not None:
        z = z + _f64(b)[None, :]
    return z.astype(out_dtype)


def topk(z: np.ndarray, k: int) -> np.ndarray:
    """Per token, the k experts with the largest logit, in the total order
    (logit descending, expert id ascending); slot j holds the j-th in that order.

    -0.0 and +0.0 compare equal (a tie, broken by id).  NaN is out of contract.
    """
    z = np.asarray(z)
    if not np.all(np.isfinite(z)):
        raise ValueError("router logits must be finite")
    T, E = z.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    ids = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary.  -z sorts the largest logit first; the
    # expert id breaks ties (lexsort is stable and compares -0.0 == +0.0).
    order = np.lexsort((ids, -z.astype(np.float64)), axis=-1)
    return order[:, :k].astype(np.int32)


def softmax_gates(sel_logits) -> np.ndarray:
    """g_j = exp(z_j) / sum_l exp(z_l) over the k selected logits (fp64).

    Equal to renormalising the full E-way softmax over the selected experts.
    """
    s = _f64(sel_logits)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True)


def topk_gates(z, idx) -> np.ndarray:
    """Renormalised softmax gates of the selected experts."""
    z = _f64(z)
    return softmax_gates(np.take_along_axis(z, np.asarray(idx, np.int64), axis=1))


# ---------------------------------------------------------------------------
# route map (device-resident routing metadata)
# ---------------------------------------------------------------------------

def route_map(idx: np.ndarray, E: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """counts[E], offsets[E+1], row_of_slot[R], slot_of_row[R] (all int32).

    counts[e]   = number of slots (t, j) routed to e
    offsets     = exclusive prefix sum of counts, offsets[E] = R = T*k
    row_of_slot = for flattened slot s = t*k + j, the row of the expert-sorted
                  buffer that holds it: offsets[e] + (number of slots s' < s
                  routed to the same expert e)
    slot_of_row = the inverse permutation

    OLMo-core 3 tutorial, "另外两处税：主机同步与 padding": counts, per-expert row
    counts and the per-expert permutation all come from the route map.
    """
    flat = np.asarray(idx).reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    R = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    # a stable sort by expert id keeps slots of one expert in ascending order
    slot_of_row = np.argsort(flat, kind="stable")
    row_of_slot = np.empty(R, np.int64)
    row_of_slot[slot_of_row] = np.arange(R)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            row_of_slot.astype(np.int32), slot_of_row.astype(np.int32))


# ---------------------------------------------------------------------------
# dispatch / expert FFN / combine
# ---------------------------------------------------------------------------

def dispatch(x, row_of_slot: np.ndarray, k: int) -> np.ndarray:
    """Xp[row_of_slot[t*k+j]] = x[t] for every token t and slot j."""
    x = _f64(x)
    T, d = x.shape
    Xp = np.empty((T * k, d))
    slots = np.arange(T * k)
    Xp[np.asarray(row_of_slot, np.int64)[slots]] = x[slots // k]
    return Xp


def silu(u: np.ndarray) -> np.ndarray:
    """silu(u) = u * sigmoid(u)."""
    return u / (1.0 + np.exp(-u))


def _sigmoid(u: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-u))


def expert_ffn_forward(Xp, offsets, W1, W3, W2) -> Dict[str, np.ndarray]:
    """Per expert e on its rows Xp[offsets[e]:offsets[e+1]]:
    H1 = X W1[e], H3 = X W3[e], A = silu(H1) * H3, Yp = A W2[e].

    One loop over experts, each on exactly its routed rows (no capacity).
    """
    Xp = _f64(Xp)
    off = np.asarray(offsets, np.int64)
    E = off.size - 1
    R = Xp.shape[0]
    h = np.asarray(W1).shape[2]
    d_out = np.asarray(W2).shape[2]
    H1 = np.zeros((R, h)); H3 = np.zeros((R, h)); A = np.zeros((R, h))
    Yp = np.zeros((R, d_out))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        X = Xp[lo:hi]
        H1[lo:hi] = X @ _f64(W1[e])
        H3[lo:hi] = X @ _f64(W3[e])
        A[lo:hi] = silu(H1[lo:hi]) * H3[lo:hi]
        Yp[lo:hi] = A[lo:hi] @ _f64(W2[e])
    return {"H1": H1, "H3": H3, "A": A, "Yp": Yp}


def combine(Yp, row_of_slot, g, k: int) -> np.ndarray:
    """out[t] = sum_j g[t,j] * Yp[row_of_slot[t*k+j]]; g = None means all ones."""
    Yp = _f64(Yp)
    rows = np.asarray(row_of_slot, np.int64).reshape(-1, k)
    T = rows.shape[0]
    out = np.zeros((T, Yp.shape[1]))
    for j in range(k):
        w = 1.0 if g is None else _f64(g)[:, j:j + 1]
        out += w * Yp[rows[:, j]]
    return out


# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------

def combine_backward(dOut, Yp, row_of_slot, g, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Gradients of out = sum_j g_j Yp[row(t,j)]:
    dYp[row(t,j)] = g[t,j] * dOut[t]   and   dg[t,j] = <dOut[t], Yp[row(t,j)]>.
    """
    dOut = _f64(dOut); Yp = _f64(Yp); g = _f64(g)
    rows = np.asarray(row_of_slot, np.int64).reshape(-1, k)
    T = rows.shape[0]
    dYp = np.zeros_like(Yp)
    dg = np.zeros((T, k))
    for j in range(k):
        dYp[rows[:, j]] = g[:, j:j + 1] * dOut
        dg[:, j] = np.einsum("td,td->t", dOut, Yp[rows[:, j]])
    return dYp, dg


def expert_ffn_backward(Xp, offsets, W1, W3, W2, H1, H3, A, dYp) -> Dict[str, np.ndarray]:
    """Backward of the per-expert SwiGLU FFN.

    dA  = dYp W2[e]^T
    dH1 = dA * H3 * silu'(H1),  silu'(u) = s(u) (1 + u (1 - s(u))),  s = sigmoid
    dH3 = dA * silu(H1)
    dXp = dH1 W1[e]^T + dH3 W3[e]^T
    dW2[e] = A_e^T dYp_e,  dW1[e] = X_e^T dH1_e,  dW3[e] = X_e^T dH3_e
    (a weight gradient is exactly zero for an expert with no rows).
    These are the Dgrad and Wgrad GEMMs of the OLMo-core 3 tutorial, section
    "一个低精度格式，同时压三个地方" (DeepSeek-V3 paragraph).
    """
    Xp = _f64(Xp); H1 = _f64(H1); H3 = _f64(H3); A = _f64(A); dYp = _f64(dYp)
    off = np.asarray(offsets, np.int64)
    E = off.size - 1
    d = Xp.shape[1]
    h = H1.shape[1]
    dXp = np.zeros_like(Xp)
    dH1 = np.zeros_like(H1); dH3 = np.zeros_like(H3)
    dW1 = np.zeros((E, d, h)); dW3 = np.zeros((E, d, h)); dW2 = np.zeros((E, h, d))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        dA = dYp[lo:hi] @ _f64(W2[e]).T
        s = _sigmoid(H1[lo:hi])
        dH1[lo:hi] = dA * H3[lo:hi] * s * (1.0 + H1[lo:hi] * (1.0 - s))
        dH3[lo:hi] = dA * H1[lo:hi] * s
        dXp[lo:hi] = dH1[lo:hi] @ _f64(W1[e]).T + dH3[lo:hi] @ _f64(W3[e]).T
        dW2[e] = A[lo:hi].T @ dYp[lo:hi]
        dW1[e] = Xp[lo:hi].T @ dH1[lo:hi]
        dW3[e] = Xp[lo:hi].T @ dH3[lo:hi]
    return {"dXp": dXp, "dH1": dH1, "dH3": dH3, "dW1": dW1, "dW3": dW3, "dW2": dW2}


def unpermute_sum(dXp, row_of_slot, k: int) -> np.ndarray:
    """dX[t] = sum_j dXp[row_of_slot[t*k+j]] (combine with unit gates)."""
    return combine(dXp, row_of_slot, None, k)


def router_topk_backward(g, dg, idx, E: int) -> np.ndarray:
    """Gradient of the renormalised top-k softmax w.r.t. the E logits:
    dz[t, idx[t,j]] = g_j (dg_j - sum_l g_l dg_l), zero for unselected experts.
    """
    g = _f64(g); dg = _f64(dg)
    idx = np.asarray(idx, np.int64)
    T, k = idx.shape
    inner = (g * dg).sum(axis=1, keepdims=True)
    dz = np.zeros((T, E))
    np.put_along_axis(dz, idx, g * (dg - inner), axis=1)
    return dz


def router_logits_backward(x, W_r, dz) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Backward of z = x W_r + b: dX = dz W_r^T, dW_r = x^T dz, db = sum_t dz."""
    x = _f64(x); W_r = _f64(W_r); dz = _f64(dz)
    return dz @ W_r.T, x.T @ dz, dz.sum(axis=0)


# ---------------------------------------------------------------------------
# whole layer
# ---------------------------------------------------------------------------

def layer_forward(inp: Dict[str, np.ndarray], k: int, E: int,
                  logits: Optional[np.ndarray] = None,
                  logits_dtype=np.float32) -> Dict[str, np.ndarray]:
    """Forward of the whole layer on one workload's inputs.

    ``logits``: optional fp32 router logits to route on (the parity tests pass
    the device's logits here so that top-k is compared on identical inputs).
    """
    res: Dict[str, np.ndarray] = {}
    if "idx" in inp:                       # synthetic uniform routing
        idx = np.asarray(inp["idx"], np.int32)
        g = softmax_gates(inp["glogit"])
    else:                                  # learned router
        z = router_logits(inp["x"], inp["W_r"], inp.get("b"), logits_dtype) \
            if logits is None else np.asarray(logits)
        res["z"] = z
        idx = topk(z, k)
        g = topk_gates(z, idx)
    counts, offsets, ros, sor = route_map(idx, E)
    Xp = dispatch(inp["x"], ros, k)
    ffn = expert_ffn_forward(Xp, offsets, inp["W1"], inp["W3"], inp["W2"])
    out = combine(ffn["Yp"], ros, g, k)
    res.update(idx=idx, g=g, counts=counts, offsets=offsets, row_of_slot=ros,
               slot_of_row=sor, Xp=Xp, out=out, **ffn)
    return res


def layer_backward(inp: Dict[str, np.ndarray], fwd: Dict[str, np.ndarray],
                   k: int, E: int) -> Dict[str, np.ndarray]:
    """Backward of the whole layer for upstream gradient inp['dY']."""
    dYp, dg = combine_backward(inp["dY"], fwd["Yp"], fwd["row_of_slot"], fwd["g"], k)
    bw = expert_ffn_backward(fwd["Xp"], fwd["offsets"], inp["W1"], inp["W3"],
                             inp["W2"], fwd["H1"], fwd["H3"], fwd["A"], dYp)
    dX = unpermute_sum(bw["dXp"], fwd["row_of_slot"], k)
    dz = router_topk_backward(fwd["g"], dg, fwd["idx"], E)
    res = dict(dYp=dYp, dg=dg, dX_expert=dX, dz=dz, **bw)
    if "W_r" in inp:
        dXr, dWr, db = router_logits_backward(inp["x"], inp["W_r"], dz)
        res.update(dX=dX + dXr, dW_r=dWr, db=db)
    else:
        # synthetic routing: gate logits are inputs, not functions of x
        res.update(dX=dX)
    return res
