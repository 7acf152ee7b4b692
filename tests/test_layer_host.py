"""Host-side logic of MoELayer that needs no GPU: the activation bytes each
backward policy keeps alive between the forward and the backward."""
from token_dispatch_grouped_router_gb300 import build as B
from token_dispatch_grouped_router_gb300.layer import MoELayer


def test_recompute_keeps_fewer_activation_bytes():
    B.build()
    T, d, E, k, h = 64, 128, 4, 2, 192
    layer = MoELayer(T, d, E, k, h, learned=False, device="cpu")
    b = layer.activation_bytes()
    R = T * k
    # the recompute policy drops exactly Xp (R x d) and H1, H3, A (R x h each), bf16
    assert b["saved"] - b["recompute"] == 2 * R * d + 3 * 2 * R * h
    # what both keep: Yp and x (bf16) and the int32 / fp32 routing tensors
    assert b["recompute"] == 2 * R * d + 2 * T * d + 4 * (3 * T * k + 2 * R + 2 * E + 1)
