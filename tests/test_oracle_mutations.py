"""Planted mistakes in the oracle (CPU only).

Each case below patches one plausible error into one oracle function -- a tie
broken the wrong way, a dropped term, a wrong sign, swapped operands, an
off-by-one -- and requires that at least one of the oracle's pins (the tests
in test_oracle_*.py, which check it against brute force, closed forms, hand
worked examples, library routines and finite differences) then fails.  This
is the evidence that the pins constrain every step they claim to pin.  The
mistakes live only here, in patched copies of the oracle's functions; the
patches are undone after each case.
"""
import numpy as np
import pytest

import oracle.layer as ol
import oracle.mxfp8 as mx
import oracle.padded as pd

import test_oracle_backward as tb
import test_oracle_ffn as tf
import test_oracle_mxfp8_padded as tm
import test_oracle_routing as tr

_ORIG = {n: getattr(ol, n) for n in (
    "topk", "route_map", "expert_ffn_forward", "combine", "combine_backward",
    "expert_ffn_backward", "dispatch", "router_logits", "unpermute_sum")}
_ORIG_MX = {n: getattr(mx, n) for n in ("block_exponent", "e4m3_decode", "dequantize_blocks")}
_ORIG_PD = {n: getattr(pd, n) for n in ("capacity_route_map",)}


def _tiny(routing):
    """The backward pins' fixture value (test_oracle_backward.py, fixture tiny)."""
    T, d, E, k, h = 6, 8, 3, 2, 12
    rng = np.random.default_rng(11)
    inp = dict(x=rng.standard_normal((T, d)),
               W1=rng.standard_normal((E, d, h)) / np.sqrt(d),
               W3=rng.standard_normal((E, d, h)) / np.sqrt(d),
               W2=rng.standard_normal((E, h, d)) / np.sqrt(h))
    if routing == "learned":
        inp["W_r"] = rng.standard_normal((d, E))
        inp["b"] = rng.standard_normal(E)
    else:
        inp["idx"] = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        inp["glogit"] = rng.standard_normal((T, k))
    dY = rng.standard_normal((T, d))
    return routing, inp, dY, k, E


# ------------------------------------------------------------------ pins
ROUTING = [lambda: tr.test_topk_brute_force_with_ties(8, 4),
           lambda: tr.test_topk_brute_force_with_ties(6, 3),
           tr.test_topk_brute_force_continuous, tr.test_topk_signed_zero_is_a_tie]
GATES = [tr.test_gates_closed_forms]
ROUTE_MAP = [tr.test_route_map_hand_worked, lambda: tr.test_route_map_brute_force(33, 4, 8)]
FFN = [tf.test_silu_matches_library, tf.test_identity_experts_dispatch_combine_exact,
       tf.test_identical_experts_reduce_to_dense_ffn, tf.test_single_expert_is_dense_swiglu,
       tf.test_gate_branch_goes_through_silu, tf.test_each_expert_uses_its_own_weights]
BACKWARD = [lambda: tb.test_backward_matches_finite_differences(_tiny("uniform")),
            lambda: tb.test_backward_matches_finite_differences(_tiny("learned")),
            tb.test_empty_expert_weight_gradient_is_exactly_zero,
            tb.test_identical_experts_gradients_sum_to_dense]
MXFP8 = [tm.test_e4m3_decode_matches_library_on_all_codes,
         tm.test_e4m3_encode_roundtrip_and_library_rounding,
         tm.test_block_exponent_is_smallest_fitting_power, tm.test_qdq_error_bound,
         tm.test_qdq_is_exact_on_representable_blocks]
PADDED = [tm.test_padded_drops_overflow_by_hand, tm.test_capacity_route_map_by_hand_and_against_the_kept_mask,
          tm.test_padded_backward_drop_by_hand]
MXFP8_GEMMS = [lambda: tm.test_mxfp8_forward_blocks_run_along_each_reduction_dimension("Xp and W1/W3"),
               lambda: tm.test_mxfp8_forward_blocks_run_along_each_reduction_dimension("A and W2"),
               tm.test_mxfp8_forward_error_matches_format_precision,
               tm.test_mxfp8_dgrad_exact_on_representable_operands_and_at_format_precision]


# --------------------------------------------------------------- mistakes
def _topk_ties_to_higher_id(z, k):
    z = np.asarray(z)
    return (z.shape[1] - 1 - _ORIG["topk"](z[:, ::-1], k)).astype(np.int32)


def _topk_smallest(z, k):
    return _ORIG["topk"](-np.asarray(z, np.float64), k)


def _gates_unnormalised(sel):
    s = np.asarray(sel, np.float64)
    return np.exp(s - s.max(axis=1, keepdims=True))


def _gates_full_softmax(z, idx):
    z = np.asarray(z, np.float64)
    e = np.exp(z - z.max(axis=1, keepdims=True))
    return np.take_along_axis(e / e.sum(axis=1, keepdims=True), np.asarray(idx, np.int64), axis=1)


def _route_map_reverse_rank(idx, E):
    c, o, ros, sor = _ORIG["route_map"](idx, E)
    flat = np.asarray(idx).reshape(-1)
    ros2 = ros.astype(np.int64).copy()
    for e in range(E):
        seg = np.nonzero(flat == e)[0]
        ros2[seg] = o[e] + (len(seg) - 1 - np.arange(len(seg)))
    sor2 = np.empty_like(ros2)
    sor2[ros2] = np.arange(ros2.size)
    return c, o, ros2.astype(np.int32), sor2.astype(np.int32)


def _route_map_inclusive_offsets(idx, E):
    c, o, ros, sor = _ORIG["route_map"](idx, E)
    o2 = np.concatenate([np.cumsum(c), [c.sum()]]).astype(np.int32)
    return c, o2, ros, sor


def _dispatch_wrong_token(x, row_of_slot, k):
    x = np.asarray(x, np.float64)
    T, d = x.shape
    Xp = np.empty((T * k, d))
    slots = np.arange(T * k)
    Xp[np.asarray(row_of_slot, np.int64)[slots]] = x[slots % T]
    return Xp


def _ffn_branches_swapped(Xp, offsets, W1, W3, W2):
    return _ORIG["expert_ffn_forward"](Xp, offsets, W3, W1, W2)


def _combine_without_gates(Yp, row_of_slot, g, k):
    return _ORIG["combine"](Yp, row_of_slot, None, k)


def _combine_bwd_without_gates(dOut, Yp, row_of_slot, g, k):
    return _ORIG["combine_backward"](dOut, Yp, row_of_slot, np.ones_like(np.asarray(g, np.float64)), k)


def _ffn_bwd_dw1_dw3_swapped(*a):
    r = dict(_ORIG["expert_ffn_backward"](*a))
    r["dW1"], r["dW3"] = r["dW3"], r["dW1"]
    return r


def _router_bwd_not_centred(g, dg, idx, E):
    g = np.asarray(g, np.float64); dg = np.asarray(dg, np.float64)
    idx = np.asarray(idx, np.int64)
    dz = np.zeros((idx.shape[0], E))
    np.put_along_axis(dz, idx, g * dg, axis=1)
    return dz


def _router_logits_bwd_dx_dropped(x, W_r, dz):
    x = np.asarray(x, np.float64); dz = np.asarray(dz, np.float64)
    return np.zeros((x.shape[0], np.asarray(W_r).shape[0])), x.T @ dz, dz.sum(axis=0)


def _capacity_keeps_last(idx, E, C):
    flat = np.asarray(idx, np.int64).reshape(-1)
    routed = np.bincount(flat, minlength=E).astype(np.int64)
    ros = np.full(flat.size, -1, np.int64)
    sor = np.full(E * C, -1, np.int64)
    seen = np.zeros(E, np.int64)
    for s, e in enumerate(flat):
        r = seen[e] - (routed[e] - min(routed[e], C))       # the last C slots stay
        seen[e] += 1
        if r >= 0:
            ros[s] = e * C + r
            sor[e * C + r] = s
    counts = np.minimum(routed, C)
    offsets = np.arange(E + 1, dtype=np.int64) * C
    return tuple(a.astype(np.int32) for a in (counts, offsets, ros, sor, routed))


def _router_logits_without_bias(x, W_r, b=None, out_dtype=np.float32):
    return _ORIG["router_logits"](x, W_r, None, out_dtype)


def _combine_bwd_dg_next_row(dOut, Yp, row_of_slot, g, k):
    dYp, _ = _ORIG["combine_backward"](dOut, Yp, row_of_slot, g, k)
    rows = np.asarray(row_of_slot, np.int64).reshape(-1, k)
    dOut = np.asarray(dOut, np.float64); Yp = np.asarray(Yp, np.float64)
    dg = np.stack([np.einsum("td,td->t", dOut, Yp[rows[:, (j + 1) % k]]) for j in range(k)], axis=1)
    return dYp, dg


def _unpermute_first_slot_only(dXp, row_of_slot, k):
    rows = np.asarray(row_of_slot, np.int64).reshape(-1, k)
    return np.asarray(dXp, np.float64)[rows[:, 0]]


def _dequantize_bias_126(q, s, axis=-1):
    return _ORIG_MX["dequantize_blocks"](q, (np.asarray(s).astype(np.int64) + 1).astype(np.uint8), axis)


def _capacity_counts_not_clamped(idx, E, C):
    counts, offsets, ros, sor, routed = _ORIG_PD["capacity_route_map"](idx, E, C)
    return routed.copy(), offsets, ros, sor, routed


def _e4m3_truncating(v):
    v = np.asarray(v, np.float64)
    pos = mx._POS_VALUES
    a = np.minimum(np.abs(v), mx.E4M3_MAX)
    code = np.searchsorted(pos, a, side="right") - 1          # round toward zero
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def _mxfp8_forward_axes(x_axis, w13_axis, a_axis, w2_axis):
    """The MXFP8 forward with each operand's blocks along the given axis (the
    oracle's are 1, 0, 1, 0: along each GEMM's reduction dimension)."""
    def fwd(Xp, offsets, W1, W3, W2):
        Xq = mx.qdq(Xp, axis=x_axis)
        off = np.asarray(offsets, np.int64)
        R, h = Xq.shape[0], np.asarray(W1).shape[2]
        H1 = np.zeros((R, h)); H3 = np.zeros((R, h)); A = np.zeros((R, h))
        Yp = np.zeros((R, np.asarray(W2).shape[2]))
        for e in range(off.size - 1):
            lo, hi = off[e], off[e + 1]
            if hi == lo:
                continue
            H1[lo:hi] = Xq[lo:hi] @ mx.qdq(W1[e], axis=w13_axis)
            H3[lo:hi] = Xq[lo:hi] @ mx.qdq(W3[e], axis=w13_axis)
            A[lo:hi] = ol.silu(H1[lo:hi]) * H3[lo:hi]
            Yp[lo:hi] = mx.qdq(A[lo:hi], axis=a_axis) @ mx.qdq(W2[e], axis=w2_axis)
        return {"H1": H1, "H3": H3, "A": A, "Yp": Yp}
    return fwd


def _mxfp8_dgrad_weights_along_d(dH1, dH3, offsets, W1, W3):
    off = np.asarray(offsets, np.int64)
    q1, q3 = mx.qdq(dH1, axis=1), mx.qdq(dH3, axis=1)
    out = np.zeros((q1.shape[0], np.asarray(W1).shape[1]))
    for e in range(off.size - 1):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            out[lo:hi] = q1[lo:hi] @ mx.qdq(W1[e], axis=0).T + q3[lo:hi] @ mx.qdq(W3[e], axis=0).T
    return out


MISTAKES = {
    # (module, attribute, replacement, pins)
    "topk: ties to the higher expert id": (ol, "topk", _topk_ties_to_higher_id, ROUTING),
    "topk: the k smallest logits": (ol, "topk", _topk_smallest, ROUTING),
    "gates: softmax not normalised": (ol, "softmax_gates", _gates_unnormalised, GATES),
    "gates: full E-way softmax, not renormalised": (ol, "topk_gates", _gates_full_softmax, GATES + BACKWARD),
    "route map: ranks in reverse slot order": (ol, "route_map", _route_map_reverse_rank, ROUTE_MAP),
    "route map: inclusive prefix sum": (ol, "route_map", _route_map_inclusive_offsets, ROUTE_MAP),
    "dispatch: token index s % T instead of s // k": (ol, "dispatch", _dispatch_wrong_token, FFN),
    "FFN: W1 and W3 swapped (silu on the wrong branch)": (ol, "expert_ffn_forward", _ffn_branches_swapped, FFN),
    "FFN: silu dropped": (ol, "silu", lambda u: u, FFN),
    "combine: gates ignored": (ol, "combine", _combine_without_gates, FFN + BACKWARD),
    "backward: sigmoid of -u in silu'": (ol, "_sigmoid", lambda u: 1.0 / (1.0 + np.exp(u)), BACKWARD),
    "backward: dW1 and dW3 swapped": (ol, "expert_ffn_backward", _ffn_bwd_dw1_dw3_swapped, BACKWARD),
    "backward: dYp without the gate": (ol, "combine_backward", _combine_bwd_without_gates, BACKWARD),
    "backward: top-k softmax Jacobian not centred": (ol, "router_topk_backward", _router_bwd_not_centred, BACKWARD),
    "backward: router term of dX dropped": (ol, "router_logits_backward", _router_logits_bwd_dx_dropped, BACKWARD),
    "MXFP8: block exponent one too large": (mx, "block_exponent", lambda amax: _ORIG_MX["block_exponent"](amax) + 1, MXFP8),
    "MXFP8: E4M3 rounding toward zero": (mx, "e4m3_encode", _e4m3_truncating, MXFP8),
    "MXFP8: subnormal step 2^-10 instead of 2^-9": (
        mx, "e4m3_decode",
        lambda c: np.where(((np.asarray(c).astype(np.int64) >> 3) & 0xF) == 0,
                           _ORIG_MX["e4m3_decode"](c) / 2, _ORIG_MX["e4m3_decode"](c)), MXFP8),
    "padded: the last C slots kept instead of the first": (pd, "capacity_route_map", _capacity_keeps_last, PADDED),
    "router logits: bias dropped": (ol, "router_logits", _router_logits_without_bias, BACKWARD),
    "combine backward: dg from the next slot's row": (ol, "combine_backward", _combine_bwd_dg_next_row, BACKWARD),
    "unpermute-sum: first slot only": (ol, "unpermute_sum", _unpermute_first_slot_only, BACKWARD),
    "MXFP8: scale byte read with bias 126": (mx, "dequantize_blocks", _dequantize_bias_126, MXFP8),
    "padded: kept counts not clamped at C": (pd, "capacity_route_map", _capacity_counts_not_clamped, PADDED),
    "MXFP8 forward: Xp blocks across rows": (mx, "expert_ffn_forward_mxfp8", _mxfp8_forward_axes(0, 0, 1, 0), MXFP8_GEMMS),
    "MXFP8 forward: W1/W3 blocks along h": (mx, "expert_ffn_forward_mxfp8", _mxfp8_forward_axes(1, 1, 1, 0), MXFP8_GEMMS),
    "MXFP8 forward: A blocks across rows": (mx, "expert_ffn_forward_mxfp8", _mxfp8_forward_axes(1, 0, 0, 0), MXFP8_GEMMS),
    "MXFP8 forward: W2 blocks along d": (mx, "expert_ffn_forward_mxfp8", _mxfp8_forward_axes(1, 0, 1, 1), MXFP8_GEMMS),
    "MXFP8 dgrad: weights in blocks along d": (mx, "expert_dgrad_dx_mxfp8", _mxfp8_dgrad_weights_along_d, MXFP8_GEMMS),
}


def _failures(pins):
    n = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            n += 1
    return n


def test_pins_pass_on_the_oracle_as_written():
    # the control: every pin used below passes without a planted mistake
    for group in (ROUTING, GATES, ROUTE_MAP, FFN, BACKWARD, MXFP8, PADDED, MXFP8_GEMMS):
        assert _failures(group) == 0


@pytest.mark.parametrize("name", list(MISTAKES))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    mod, attr, repl, pins = MISTAKES[name]
    monkeypatch.setattr(mod, attr, repl)
    assert _failures(pins) >= 1, f"no pin caught: {name}"
