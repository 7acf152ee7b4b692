"""Pins for the oracle's dispatch, expert FFN and combine (CPU only)."""
import numpy as np
import pytest
import torch

from oracle import layer as ol
from token_dispatch_grouped_router_gb300 import workloads as wl


def _rand_layer(T, d, E, k, h, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, d, h)) / np.sqrt(d)
    W3 = rng.standard_normal((E, d, h)) / np.sqrt(d)
    W2 = rng.standard_normal((E, h, d)) / np.sqrt(h)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    glog = rng.standard_normal((T, k))
    return x, W1, W3, W2, idx, glog


def test_silu_matches_library():
    u = np.linspace(-30, 30, 2001)
    ref = torch.nn.functional.silu(torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(ol.silu(u), ref, rtol=1e-14, atol=1e-300)


def test_identity_experts_dispatch_combine_exact():
    # Yp = Xp (identity experts) and unit gates give out = k * x exactly: every
    # routed row goes out and comes back exactly once.
    rng = np.random.default_rng(3)
    T, d, E, k = 40, 16, 6, 3
    x = wl.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    _, _, ros, _ = ol.route_map(idx, E)
    Xp = ol.dispatch(x, ros, k)
    out = ol.combine(Xp, ros, np.ones((T, k)), k)
    assert np.array_equal(out, k * ol.decode_bf16(x))
    # one-hot routing (k = 1) is a plain gather back to token order
    idx1 = rng.integers(0, E, (T, 1))
    _, off1, ros1, sor1 = ol.route_map(idx1, E)
    Xp1 = ol.dispatch(x, ros1, 1)
    assert np.array_equal(Xp1, ol.decode_bf16(x)[sor1])


def test_identical_experts_reduce_to_dense_ffn():
    T, d, E, k, h = 24, 16, 5, 2, 12
    x, W1, W3, W2, idx, glog = _rand_layer(T, d, E, k, h, seed=4)
    W1[:] = W1[0]; W3[:] = W3[0]; W2[:] = W2[0]
    g = ol.softmax_gates(glog)
    _, offsets, ros, _ = ol.route_map(idx, E)
    Yp = ol.expert_ffn_forward(ol.dispatch(x, ros, k), offsets, W1, W3, W2)["Yp"]
    out = ol.combine(Yp, ros, g, k)
    # dense SwiGLU FFN of every token through torch's matmul and silu
    xt = torch.from_numpy(x)
    dense = (torch.nn.functional.silu(xt @ torch.from_numpy(W1[0]))
             * (xt @ torch.from_numpy(W3[0]))) @ torch.from_numpy(W2[0])
    np.testing.assert_allclose(out, dense.numpy(), rtol=1e-12, atol=1e-12)
    # with arbitrary (unnormalised) gates the result scales by the gate sum
    graw = np.abs(glog) + 0.1
    out2 = ol.combine(Yp, ros, graw, k)
    np.testing.assert_allclose(out2, dense.numpy() * graw.sum(1, keepdims=True),
                               rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_swiglu():
    T, d, E, k, h = 10, 8, 1, 1, 6
    x, W1, W3, W2, idx, glog = _rand_layer(T, d, E, k, h, seed=5)
    inp = dict(x=x, W1=W1, W3=W3, W2=W2, idx=idx, glogit=glog)
    out = ol.layer_forward(inp, k, E)["out"]
    xt = torch.from_numpy(x)
    dense = (torch.nn.functional.silu(xt @ torch.from_numpy(W1[0]))
             * (xt @ torch.from_numpy(W3[0]))) @ torch.from_numpy(W2[0])
    np.testing.assert_allclose(out, dense.numpy(), rtol=1e-12, atol=1e-12)


def test_gate_branch_goes_through_silu():
    # W1 is the silu branch: drive X W1 far negative and the output vanishes
    # whatever W3 is; drive X W3 far negative instead and it does not.
    T, d, E, k, h = 6, 4, 2, 1, 3
    rng = np.random.default_rng(6)
    x = np.abs(rng.standard_normal((T, d))) + 0.5
    big = -np.full((E, d, h), 50.0)
    other = rng.standard_normal((E, d, h))
    W2 = rng.standard_normal((E, h, d))
    idx = rng.integers(0, E, (T, 1))
    _, off, ros, _ = ol.route_map(idx, E)
    Xp = ol.dispatch(x, ros, 1)
    y_w1neg = ol.expert_ffn_forward(Xp, off, big, other, W2)["Yp"]
    y_w3neg = ol.expert_ffn_forward(Xp, off, other, big, W2)["Yp"]
    assert np.max(np.abs(y_w1neg)) < 1e-30
    assert np.max(np.abs(y_w3neg)) > 1e-3


def test_each_expert_uses_its_own_weights():
    # routing every token to expert e must equal the dense FFN with W[e]
    T, d, E, k, h = 9, 8, 4, 1, 5
    x, W1, W3, W2, _, _ = _rand_layer(T, d, E, k, h, seed=7)
    for e in range(E):
        idx = np.full((T, 1), e)
        inp = dict(x=x, W1=W1, W3=W3, W2=W2, idx=idx, glogit=np.zeros((T, 1)))
        out = ol.layer_forward(inp, 1, E)["out"]
        ref = (ol.silu(x @ W1[e]) * (x @ W3[e])) @ W2[e]
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_workload_generator_shapes_and_stats():
    w = wl.small_workload(T=256, d=64, E=8, k=4, h=32)
    a = wl.generate(w, seed=0)
    b = wl.generate(w, seed=0)
    for key in a:
        assert np.array_equal(a[key], b[key])          # seeded
    assert a["x"].dtype == np.uint16 and a["x"].shape == (256, 64)
    assert a["W2"].shape == (8, 32, 64)
    idx = a["idx"]
    assert idx.shape == (256, 4) and idx.min() >= 0 and idx.max() < 8
    assert all(len(set(r)) == 4 for r in idx)           # distinct experts
    # bf16 rounding is nearest-even: the error is at most half a bf16 ulp
    v = np.random.default_rng(9).standard_normal(10000).astype(np.float32)
    r = ol.decode_bf16(wl.bf16_bits(v))
    ulp = np.exp2(np.floor(np.log2(np.abs(v.astype(np.float64)))) - 7)
    assert np.all(np.abs(r - v) <= ulp / 2)
    # a different seed changes the draw
    c = wl.generate(w, seed=1)
    assert not np.array_equal(a["x"], c["x"])


def test_zipf_workload_is_skewed():
    # the skewed recipe at the full pool (E=128) on a reduced token count:
    # some experts receive nothing and the hottest is far above the mean
    w = wl.small_workload(T=2048, d=256, E=128, k=4, h=64, routing="learned", zipf=True)
    a = wl.generate(w, seed=0, with_backward=False)
    z = ol.router_logits(a["x"], a["W_r"], a["b"])
    counts = ol.route_map(ol.topk(z, 4), 128)[0]
    assert (counts == 0).sum() >= 1
    assert counts.max() > 4 * counts.mean()
