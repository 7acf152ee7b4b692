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


def test_mxfp8_saved_activations_keep_codes_and_scales():
    B.build()
    T, d, E, k, h = 64, 128, 4, 2, 192
    layer = MoELayer(T, d, E, k, h, learned=False, device="cpu")
    b = layer.activation_bytes()
    R = T * k
    # Xp and A go from bf16 (2 bytes) to one E4M3 byte plus one scale byte per
    # 32 values; H1 and H3 stay bf16
    assert b["saved"] - b["mxfp8_saved"] == (2 * R * d - (R * d + R * d // 32)) + \
        (2 * R * h - (R * h + R * h // 32))
    assert b["recompute"] < b["mxfp8_saved"] < b["saved"]


def test_bench_capacity_stats_by_hand():
    # 3 experts, T*k = 12 routed rows, capacity ceil(1.25 * 12 / 3) = 5:
    # loads 9, 3, 0 drop 4 rows; the padded layer multiplies 15 rows for 12
    import bench
    st = bench.capacity_stats([9, 3, 0], T=6, k=2, E=3)
    assert st["capacity"] == 5 and st["dropped_rows"] == 4
    assert abs(st["dropped_fraction"] - 4 / 12) < 1e-12
    assert abs(st["padded_over_routed_rows"] - 15 / 12) < 1e-12
    # enough capacity: nothing dropped
    assert bench.capacity_stats([4, 4, 4], T=6, k=2, E=3)["dropped_rows"] == 0


class _FakeEvent:
    """A recorded CUDA event stand-in: a timestamp in ms."""
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_bench_step_timings_per_stream():
    import bench
    E = _FakeEvent
    # one step: main stream 1 (a, wgrad, join, end), second stream 2 (unpermute, side_end)
    step = [("a", E(0.0), 1), ("wgrad", E(1.0), 1), ("join", E(3.0), 1),
            ("unpermute", E(1.2), 2), ("side_end", E(2.0), 2), ("end", E(3.5), 1)]
    step_ms, per_label, side = bench.step_timings([step, step])
    assert step_ms == [3.5, 3.5]                       # first to last mark of stream 1
    assert per_label["a"] == [1.0, 1.0]
    assert per_label["wgrad"] == [2.0, 2.0]            # to the next mark on its own stream
    assert per_label["join"] == [0.5, 0.5]
    assert per_label["unpermute"] == [0.8, 0.8]        # measured on stream 2 alone
    assert "side_end" not in per_label and "end" not in per_label
    assert side == {"unpermute", "side_end"}
    # one stream: consecutive marks
    step_ms, per_label, side = bench.step_timings([[("x", E(0.0), 7), ("y", E(0.25), 7), ("end", E(1.0), 7)]])
    assert step_ms == [1.0] and per_label == {"x": [0.25], "y": [0.75]} and side == set()
