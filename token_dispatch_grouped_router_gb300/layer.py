"""The MoE expert layer as a sequence of libmoe calls on preallocated buffers.

``MoELayer`` owns the device buffers of one layer step (PyTorch supplies the
memory and the stream) and runs forward and backward purely through the C-ABI
entry points:

forward : [router_logits ->] router_topk | router_gates -> expert_offsets ->
          dispatch_rows -> grouped_swiglu_fwd (up, down) -> combine
backward: [dispatch_rows -> grouped_swiglu_fwd_up (recompute)] -> combine_bwd ->
          grouped_swiglu_bwd (dact, dx, wgrad) -> combine(gates = None) ->
          router_topk_bwd [-> router_logits_bwd]

With ``recompute=True`` the backward does not use the expert rows Xp or the
SwiGLU intermediates H1, H3, A left by the forward: it gathers the rows again
from x and recomputes H1, H3, A from them, so that only x, the routing and Yp
(for the gate gradient) have to live from the forward to the backward.

With ``capacity_factor=f`` the layer is the capacity-padded alternative the
device route map replaces: every expert gets C = ceil(f * T * k / E) rows of
the expert-sorted buffers (its first C routed slots in token order, then zero
rows), later slots are dropped, and the same grouped GEMMs run on all E * C
rows (the ``_capacity`` route-map, dispatch and combine calls).

With ``side_stream=True`` the combine(gates = None) and the router backward
run on a second stream beside the wgrad GEMM, joined before the step ends
(same results bit for bit; off by default: with steps queued back to back it
was not faster).

Nothing is copied back to the host and nothing waits on the host.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np
import torch

from . import libmoe as L


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns (numpy) -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 bit patterns (numpy, host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _nomark(label: str) -> None:
    return None


class MoELayer:
    """Buffers and call sequence of one MoE layer step on one GPU."""

    def __init__(self, T: int, d: int, E: int, k: int, h: int, learned: bool,
                 device="cuda", with_backward: bool = True, recompute: bool = False,
                 capacity_factor: Optional[float] = None, side_stream: bool = False):
        self.T, self.d, self.E, self.k, self.h = T, d, E, k, h
        self.learned = learned
        self.with_backward = with_backward
        self.recompute = recompute
        # capacity-padded layer: E * C rows in every expert-sorted buffer
        self.C = int(math.ceil(capacity_factor * T * k / E)) if capacity_factor else None
        if self.C is not None:
            self.C = max(self.C, 1)           # T = 0: one zero row an expert, dW = 0
        self.R = T * k if self.C is None else E * self.C
        dev = torch.device(device)
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        e = lambda *s, dt=bf: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        R = self.R
        self.x = e(T, d)
        self.W1 = e(E, d, h); self.W3 = e(E, d, h); self.W2 = e(E, h, d)
        if learned:
            self.W_r = e(d, E, dt=f32)
            self.b: Optional[torch.Tensor] = None
            self.logits = e(T, E, dt=f32)
            self.logits_given = False
        else:
            self.glogit = e(T, k, dt=f32)
        self.idx = e(T, k, dt=i32)
        self.gate = e(T, k, dt=f32)
        self.counts = e(E, dt=i32)
        self.offsets = e(E + 1, dt=i32)
        self.row_of_slot = e(T * k, dt=i32)
        self.slot_of_row = e(R, dt=i32)
        if self.C is not None:
            self.routed = e(E, dt=i32)          # rows routed before the capacity cut
            if learned and with_backward:
                # the router backward sums over every routed slot, dropped ones
                # included: it reads the unpadded route map
                self.u_counts = e(E, dt=i32); self.u_offsets = e(E + 1, dt=i32)
                self.u_row_of_slot = e(T * k, dt=i32); self.u_slot_of_row = e(T * k, dt=i32)
        self.xp = e(R, d)
        self.h1 = e(R, h); self.h3 = e(R, h); self.a = e(R, h)
        self.yp = e(R, d)
        self.out = e(T, d)
        ws_bytes = L.moe_workspace_size(T, E, k, d, h)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        if with_backward:
            self.dY = e(T, d)
            self.dyp = e(R, d); self.dgate = e(T, k, dt=f32)
            self.dh1 = e(R, h); self.dh3 = e(R, h); self.dxp = e(R, d)
            self.dW1 = e(E, d, h); self.dW3 = e(E, d, h); self.dW2 = e(E, h, d)
            self.dX = e(T, d)
            self.dlogits = e(T, E, dt=f32)
            if learned:
                self.dW_r = e(d, E, dt=f32)
                self.db = e(E, dt=f32)
            # the backward's optional second stream (see backward); off by
            # default: with steps queued back to back it made the step slower
            self._side = None
            if side_stream and dev.type == "cuda":
                self._side = torch.cuda.Stream(device=dev)
                self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()

    # ------------------------------------------------------------- inputs
    def load_inputs(self, inp: Dict[str, np.ndarray]) -> None:
        """Copy one workload's host inputs (see workloads.generate) to the device."""
        dev = self.x.device
        self.x.copy_(bf16_tensor(inp["x"], dev))
        self.W1.copy_(bf16_tensor(inp["W1"], dev))
        self.W3.copy_(bf16_tensor(inp["W3"], dev))
        self.W2.copy_(bf16_tensor(inp["W2"], dev))
        if self.learned:
            self.W_r.copy_(torch.from_numpy(inp["W_r"]))
            if inp.get("b") is not None:
                self.b = torch.from_numpy(inp["b"]).to(dev)
        else:
            self.idx.copy_(torch.from_numpy(inp["idx"]))
            self.glogit.copy_(torch.from_numpy(inp["glogit"]))
        if self.with_backward and "dY" in inp:
            self.dY.copy_(bf16_tensor(inp["dY"], dev))

    def load_logits(self, z: np.ndarray) -> None:
        """Route on these fp32 logits instead of computing x @ W_r + b (the
        top-k and everything after it still run on the device)."""
        self.logits.copy_(torch.from_numpy(np.ascontiguousarray(z, np.float32)))
        self.logits_given = True

    # ------------------------------------------------------------ forward
    # `mark(label)` (optional) is called before each library call and with
    # "end" after the last one; the benchmark records CUDA events there.
    def route(self, mark=None) -> None:
        mark = mark or _nomark
        if self.learned:
            if not self.logits_given:
                mark("router_logits")
                L.moe_router_logits_tc(self.x, self.W_r, self.b, self.logits, self.ws)
            mark("router_topk")
            L.moe_router_topk(self.logits, self.k, self.idx, self.gate)
        else:
            mark("router_gates")
            L.moe_router_gates(self.glogit, self.gate)
        mark("expert_offsets")
        if self.C is not None:
            L.moe_expert_offsets_capacity(self.idx, self.E, self.C, self.counts, self.offsets,
                                          self.row_of_slot, self.slot_of_row, self.ws, self.routed)
        else:
            L.moe_expert_offsets(self.idx, self.E, self.counts, self.offsets, self.row_of_slot,
                                 self.slot_of_row, self.ws)

    def _combine(self, rows, gate, out) -> None:
        if self.C is not None:
            L.moe_combine_capacity(rows, self.E, self.C, self.row_of_slot, gate, self.k, out)
        else:
            L.moe_combine(rows, self.row_of_slot, gate, self.k, out)

    def forward(self, mark=None) -> torch.Tensor:
        mark = mark or _nomark
        self.route(mark)
        mark("dispatch")
        if self.C is not None:
            L.moe_dispatch_rows_capacity(self.x, self.row_of_slot, self.counts, self.k, self.C,
                                         self.xp)
        else:
            L.moe_dispatch_rows(self.x, self.row_of_slot, self.k, self.xp)
        mark("gemm_up")
        L.moe_grouped_swiglu_fwd_up(self.xp, self.offsets, self.W1, self.W3, self.h1, self.h3,
                                    self.a, self.ws)
        mark("gemm_down")
        L.moe_grouped_swiglu_fwd_down(self.a, self.offsets, self.W2, self.yp, self.ws)
        mark("combine")
        self._combine(self.yp, self.gate, self.out)
        return self.out

    # ----------------------------------------------------------- backward
    def backward(self, mark=None) -> None:
        mark = mark or _nomark
        if self.recompute and self.C is not None:
            raise ValueError("the recompute policy is not combined with capacity padding")
        if self.recompute:
            mark("dispatch_recompute")
            L.moe_dispatch_rows(self.x, self.row_of_slot, self.k, self.xp)
            mark("gemm_up_recompute")
            L.moe_grouped_swiglu_fwd_up(self.xp, self.offsets, self.W1, self.W3, self.h1,
                                        self.h3, self.a, self.ws)
        mark("combine_bwd")
        if self.C is not None:
            L.moe_combine_bwd_capacity(self.dY, self.yp, self.C, self.row_of_slot, self.counts,
                                       self.gate, self.k, self.dyp, self.dgate)
        else:
            L.moe_combine_bwd(self.dY, self.yp, self.row_of_slot, self.gate, self.k,
                              self.dyp, self.dgate)
        mark("gemm_dact")
        if getattr(self, "mx_dgrad", False):
            # dh1, dh3 also leave quantised along h for the MXFP8 dgrad
            L.moe_grouped_swiglu_bwd_dact_mxfp8(self.offsets, self.W2, self.h1, self.h3, self.dyp,
                                                self.dh1, self.dh3, self.dh1q, self.dh1s,
                                                self.dh3q, self.dh3s, self.ws)
        else:
            L.moe_grouped_swiglu_bwd_dact(self.offsets, self.W2, self.h1, self.h3, self.dyp,
                                          self.dh1, self.dh3, self.ws)
        if getattr(self, "mx_dgrad", False):
            # the block-scaled dgrad GEMM on the dact epilogue's quantised dh1, dh3
            mark("gemm_dx_mxfp8")
            L.moe_grouped_swiglu_bwd_dx_mxfp8(self.dh1q, self.dh1s, self.dh3q, self.dh3s,
                                              self.offsets, self.w1q_h, self.w3q_h,
                                              self.dx_atoms, self.dxp, self.ws)
        else:
            mark("gemm_dx")
            L.moe_grouped_swiglu_bwd_dx(self.offsets, self.W1, self.W3, self.dh1, self.dh3,
                                        self.dxp, self.ws)
        mark("gemm_wgrad")
        side = self._side
        if side is None:
            L.moe_grouped_swiglu_bwd_wgrad(self.xp, self.offsets, self.a, self.dyp, self.dh1,
                                           self.dh3, self.dW1, self.dW3, self.dW2, self.ws)
            self._unpermute_and_router_bwd(mark, logits_bwd=True)
            return
        # The unpermute, the router backward through the top-k and, for a
        # learned router without capacity padding, the router logits backward
        # read nothing the weight-gradient GEMM writes and use a part of the
        # workspace it does not, so they run on a second stream beside it, in
        # what its one block an SM leaves free (registers, threads, a few KB of
        # shared memory).  The padded layer's unpadded route map reuses the
        # GEMM's part of the workspace and waits for it.
        main = torch.cuda.current_stream(self.dX.device)
        self._fork.record(main)
        L.moe_grouped_swiglu_bwd_wgrad(self.xp, self.offsets, self.a, self.dyp, self.dh1,
                                       self.dh3, self.dW1, self.dW3, self.dW2, self.ws)
        mark("join_side")
        side.wait_event(self._fork)
        with torch.cuda.stream(side):
            self._unpermute_and_router_bwd(mark, logits_bwd=self.C is None)
            mark("side_end")
            self._join.record(side)
        main.wait_event(self._join)
        if self.learned and self.C is not None:
            self._router_logits_bwd(mark)

    def _unpermute_and_router_bwd(self, mark, logits_bwd: bool) -> None:
        mark("unpermute")
        self._combine(self.dxp, None, self.dX)
        mark("router_bwd")
        L.moe_router_topk_bwd(self.gate, self.dgate, self.idx, self.E, self.dlogits)
        if self.learned and logits_bwd:
            self._router_logits_bwd(mark)

    def _router_logits_bwd(self, mark) -> None:
        offsets, slot_of_row = self.offsets, self.slot_of_row
        if self.C is not None:
            mark("expert_offsets_unpadded")
            L.moe_expert_offsets(self.idx, self.E, self.u_counts, self.u_offsets,
                                 self.u_row_of_slot, self.u_slot_of_row, self.ws)
            offsets, slot_of_row = self.u_offsets, self.u_slot_of_row
        mark("router_logits_bwd")
        L.moe_router_logits_bwd_topk(self.x, self.W_r, self.dlogits, self.idx, offsets,
                                     slot_of_row, self.dX, self.dW_r, self.db, self.ws)

    # ------------------------------------------------------------- MXFP8
    def enable_mxfp8(self) -> None:
        """Allocate the MXFP8 buffers: K-major E4M3 weight copies with their
        E8M0 scales, quantised expert rows and quantised activations."""
        if self.C is not None:
            raise ValueError("the MXFP8 path is not combined with capacity padding")
        E, d, h, R = self.E, self.d, self.h, self.R
        dev = self.x.device
        u = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)  # noqa: E731
        self.w1q, self.w1s = u(E, h, d), u(E, h, d // 32)
        self.w3q, self.w3s = u(E, h, d), u(E, h, d // 32)
        self.w2q, self.w2s = u(E, d, h), u(E, d, h // 32)
        self.w_atoms = u(L.moe_mxfp8_weight_atom_bytes(E, d, h))
        self.xq, self.xs = u(R, d), u(R, d // 32)
        self.aq, self.as_ = u(R, h), u(R, h // 32)
        # MXFP8 dgrad: W1 / W3 quantised along h (their own copies) and the
        # quantised dh1 / dh3 of a step
        self.w1q_h, self.w1s_h = u(E, d, h), u(E, d, h // 32)
        self.w3q_h, self.w3s_h = u(E, d, h), u(E, d, h // 32)
        self.dx_atoms = u(L.moe_mxfp8_dx_weight_atom_bytes(E, d, h))
        if self.with_backward:
            self.dh1q, self.dh1s = u(R, h), u(R, h // 32)
            self.dh3q, self.dh3s = u(R, h), u(R, h // 32)
        self.mx_dgrad = False

    def quantize_weights(self, mark=None, dgrad: bool = True) -> None:
        """Re-make the MXFP8 weight copies (once per optimizer step); dgrad
        also makes the dgrad GEMM's copies of W1 / W3 (quantised along h)."""
        mark = mark or _nomark
        mark("mx_quantize_weights")
        L.moe_mxfp8_quantize_weights(self.W1, self.w1q, self.w1s)
        L.moe_mxfp8_quantize_weights(self.W3, self.w3q, self.w3s)
        L.moe_mxfp8_quantize_weights(self.W2, self.w2q, self.w2s)
        L.moe_mxfp8_weight_scale_atoms(self.w1s, self.w3s, self.w2s, self.w_atoms)
        if dgrad:
            self._quantize_dgrad_weights()

    def _quantize_dgrad_weights(self) -> None:
        """W1 and W3 quantised along h (the dgrad GEMM's reduction), from the
        bf16 weights, and their scale atoms."""
        E, d, h = self.E, self.d, self.h
        L.moe_mxfp8_quantize_rows(self.W1.view(E * d, h), self.w1q_h.view(E * d, h),
                                  self.w1s_h.view(E * d, h // 32))
        L.moe_mxfp8_quantize_rows(self.W3.view(E * d, h), self.w3q_h.view(E * d, h),
                                  self.w3s_h.view(E * d, h // 32))
        L.moe_mxfp8_dx_weight_scale_atoms(self.w1s_h, self.w3s_h, self.dx_atoms)

    def quantize_weights_from_masters(self, W1m: torch.Tensor, W3m: torch.Tensor,
                                      W2m: torch.Tensor) -> None:
        """Re-make the MXFP8 weight copies from fp32 master weights (shapes of
        W1, W3, W2): one rounding instead of fp32 -> bf16 -> E4M3."""
        L.moe_mxfp8_quantize_weights_f32(W1m, self.w1q, self.w1s)
        L.moe_mxfp8_quantize_weights_f32(W3m, self.w3q, self.w3s)
        L.moe_mxfp8_quantize_weights_f32(W2m, self.w2q, self.w2s)
        L.moe_mxfp8_weight_scale_atoms(self.w1s, self.w3s, self.w2s, self.w_atoms)
        self._quantize_dgrad_weights()

    def forward_mxfp8(self, mark=None, saved: str = "bf16") -> torch.Tensor:
        """Forward with MXFP8 GEMM operands.  saved="bf16": h1, h3, a and xp
        are also written in bf16 for the bf16 backward.  saved="mxfp8": the
        expert rows and the SwiGLU activation are kept only quantised (xq/xs,
        aq/as); ``restore_saved_mxfp8`` dequantises them for the backward."""
        if saved not in ("bf16", "mxfp8"):
            raise ValueError(f"saved must be 'bf16' or 'mxfp8', not {saved!r}")
        mark = mark or _nomark
        keep_bf16 = saved == "bf16"
        self.route(mark)
        mark("dispatch_mxfp8")
        L.moe_dispatch_rows_mxfp8(self.x, self.row_of_slot, self.k, self.xq, self.xs,
                                  self.xp if keep_bf16 else None)
        mark("gemm_fwd_mxfp8")
        L.moe_grouped_swiglu_fwd_mxfp8(self.xq, self.xs, self.offsets, self.w1q, self.w3q,
                                       self.w2q, self.w_atoms, self.h1, self.h3,
                                       self.a if keep_bf16 else None, self.aq, self.as_, self.yp,
                                       self.ws)
        mark("combine")
        L.moe_combine(self.yp, self.row_of_slot, self.gate, self.k, self.out)
        return self.out

    def restore_saved_mxfp8(self, mark=None) -> None:
        """bf16 Xp and A for the backward from their MXFP8 forms (each value is
        code * 2^(scale - 127), exact in bf16 for these magnitudes)."""
        mark = mark or _nomark
        mark("mx_dequantize_saved")
        L.moe_mxfp8_dequantize_rows(self.xq, self.xs, self.xp)
        L.moe_mxfp8_dequantize_rows(self.aq, self.as_, self.a)

    def step_mxfp8(self, mark=None, requantize: bool = True, saved: str = "bf16",
                   dgrad: str = "bf16") -> None:
        """Forward through the block-scaled GEMMs; backward in bf16, with the
        dgrad GEMM in MXFP8 too when dgrad="mxfp8"."""
        if dgrad not in ("bf16", "mxfp8"):
            raise ValueError(f"dgrad must be 'bf16' or 'mxfp8', not {dgrad!r}")
        if requantize:
            self.quantize_weights(mark, dgrad=dgrad == "mxfp8")
        self.forward_mxfp8(mark, saved=saved)
        if self.with_backward:
            if saved == "mxfp8":
                self.restore_saved_mxfp8(mark)
            self.mx_dgrad = dgrad == "mxfp8"
            try:
                self.backward(mark)
            finally:
                self.mx_dgrad = False
        if mark is not None:
            mark("end")

    def step(self, mark=None) -> None:
        self.forward(mark)
        if self.with_backward:
            self.backward(mark)
        if mark is not None:
            mark("end")

    def activation_bytes(self) -> Dict[str, int]:
        """Bytes the forward leaves for the backward, by policy: the expert
        rows Xp and H1, H3, A in bf16 ("saved"); Xp and A as MXFP8 codes with
        their scales and H1, H3 in bf16 ("mxfp8_saved"); none of them
        ("recompute").  Yp, the routing and x are kept in every policy."""
        R, d, h, T, k, E = self.R, self.d, self.h, self.T, self.k, self.E
        common = 2 * R * d + 2 * T * d + 4 * (3 * T * k + 2 * R + 2 * E + 1)
        mx = R * d + R * d // 32 + R * h + R * h // 32
        return {"saved": common + 2 * R * d + 3 * 2 * R * h,
                "mxfp8_saved": common + mx + 2 * 2 * R * h,
                "recompute": common}


class HostPipeline:
    """Layer steps fed from and drained to (pinned) host memory, with the
    host-to-device copy of step i+1's inputs and the device-to-host copy of
    step i-1's results running on their own streams while step i computes.

    The named input and output tensors of the layer get a second device copy
    and the steps alternate between the two; every other buffer of the layer
    is used by one step at a time, in stream order.  A slot's inputs are
    overwritten only after the step that read them has finished, and its
    outputs only after they have been copied out.
    """

    def __init__(self, layer: MoELayer, input_names=("x", "dY", "idx", "glogit"),
                 output_names=("out", "dX")):
        self.layer = layer
        self.inputs = [n for n in input_names if hasattr(layer, n)]
        self.outputs = list(output_names)
        names = self.inputs + self.outputs
        self.slots = [{n: getattr(layer, n) for n in names},
                      {n: torch.empty_like(getattr(layer, n)) for n in names}]
        self.h2d = torch.cuda.Stream(device=layer.x.device)
        self.d2h = torch.cuda.Stream(device=layer.x.device)

    def _use(self, slot: int) -> None:
        for n, t in self.slots[slot].items():
            setattr(self.layer, n, t)

    def run(self, host_inputs, host_outputs, before_step=None) -> None:
        """Run len(host_inputs) steps: host_inputs[i] maps input names to the
        host tensors of step i, host_outputs[i] maps output names to host
        tensors that receive step i's results.  `before_step()`, if given, is
        enqueued on the compute stream before each step.  Returns when every
        copy has been issued; the caller synchronises."""
        compute = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]
        start = torch.cuda.Event()
        start.record(compute)
        self.h2d.wait_event(start)
        try:
            for i, (hin, hout) in enumerate(zip(host_inputs, host_outputs)):
                s = i % 2
                dev = self.slots[s]
                with torch.cuda.stream(self.h2d):
                    if i >= 2:
                        self.h2d.wait_event(ev_done[s])      # step i-2 has read this slot
                    for n in self.inputs:
                        dev[n].copy_(hin[n], non_blocking=True)
                    ev_in[s].record(self.h2d)
                compute.wait_event(ev_in[s])
                if i >= 2:
                    compute.wait_event(ev_out[s])            # step i-2's results are out
                self._use(s)
                if before_step is not None:
                    before_step()
                self.layer.step()
                ev_done[s].record(compute)
                with torch.cuda.stream(self.d2h):
                    self.d2h.wait_event(ev_done[s])
                    for n in self.outputs:
                        hout[n].copy_(dev[n], non_blocking=True)
                    ev_out[s].record(self.d2h)
            for s in range(min(2, len(host_inputs))):
                compute.wait_event(ev_out[s])
        finally:
            self._use(0)
