"""Helpers shared by the GPU parity tests (not a test module).

Tolerance (floating point vs the fp64 oracle, bf16 path): relative L2 error
<= 1e-2 and max-abs error <= 3e-2 * max|ref|.  Integer outputs are compared
bit-exactly.
"""
import numpy as np
import torch

import __graft_entry__
import oracle.layer as ol
from token_dispatch_grouped_router_gb300.layer import MoELayer, bf16_bits

REL_L2 = 1e-2
MAX_ABS = 3e-2


def ensure_built():
    __graft_entry__.build()


def as_f64(t) -> np.ndarray:
    """Device tensor (bf16 / f32) -> float64 numpy."""
    if isinstance(t, torch.Tensor):
        if t.dtype == torch.bfloat16:
            return ol.decode_bf16(bf16_bits(t))
        return t.detach().cpu().numpy().astype(np.float64)
    return np.asarray(t, np.float64)


def assert_close(got, ref, name="", rel_l2=REL_L2, max_abs=MAX_ABS):
    got = as_f64(got)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    nref = np.linalg.norm(ref)
    err = np.linalg.norm(got - ref)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if nref == 0:
        assert err == 0, f"{name}: expected zeros, error {err}"
        return
    r = err / nref
    m = np.max(np.abs(got - ref))
    assert r <= rel_l2, f"{name}: rel-L2 {r:.3e} > {rel_l2}"
    assert m <= max_abs * scale, f"{name}: max-abs {m:.3e} > {max_abs} * {scale:.3e}"


def run_layer(w, inp, device="cuda", backward=True):
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=(w.routing == "learned"),
                     device=device, with_backward=backward)
    layer.load_inputs(inp)
    L = __import__("token_dispatch_grouped_router_gb300.libmoe", fromlist=["x"])
    L.moe_reset_status(layer.ws)
    if backward:
        layer.step()
    else:
        layer.forward()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    return layer


def i32(t) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.int64)
