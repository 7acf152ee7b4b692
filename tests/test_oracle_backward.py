"""Pins for the oracle's backward: fp64 central finite differences (CPU only).

The scalar loss is L = sum(dY * out); every analytic gradient of
``oracle.layer.layer_backward`` is compared with (L(p+eps) - L(p-eps)) / 2eps
of the oracle's own forward.  Shapes use d != h so a transposed operand fails.
"""
import numpy as np
import pytest

from oracle import layer as ol

EPS = 1e-6


def _loss(inp, k, E, dY):
    out = ol.layer_forward(inp, k, E, logits_dtype=np.float64)["out"]
    return float((out * dY).sum())


def _fd_check(inp, key, grad, k, E, dY, n_samples=40, seed=0):
    rng = np.random.default_rng(seed)
    arr = inp[key]
    flat_idx = rng.choice(arr.size, size=min(n_samples, arr.size), replace=False)
    ref_idx = ol.layer_forward(inp, k, E, logits_dtype=np.float64).get("idx")
    checked = 0
    for fi in flat_idx:
        pos = np.unravel_index(fi, arr.shape)
        orig = arr[pos]
        arr[pos] = orig + EPS
        fp = ol.layer_forward(inp, k, E, logits_dtype=np.float64)
        lp = float((fp["out"] * dY).sum())
        arr[pos] = orig - EPS
        fm = ol.layer_forward(inp, k, E, logits_dtype=np.float64)
        lm = float((fm["out"] * dY).sum())
        arr[pos] = orig
        if ref_idx is not None and not (np.array_equal(fp["idx"], ref_idx)
                                        and np.array_equal(fm["idx"], ref_idx)):
            continue            # the perturbation crossed a routing boundary
        num = (lp - lm) / (2 * EPS)
        assert abs(num - grad[pos]) <= 1e-6 * max(1.0, abs(num)), (key, pos, num, grad[pos])
        checked += 1
    assert checked >= min(n_samples, arr.size) // 2


@pytest.fixture(params=["learned", "uniform"])
def tiny(request):
    T, d, E, k, h = 6, 8, 3, 2, 12
    rng = np.random.default_rng(11)
    inp = dict(x=rng.standard_normal((T, d)),
               W1=rng.standard_normal((E, d, h)) / np.sqrt(d),
               W3=rng.standard_normal((E, d, h)) / np.sqrt(d),
               W2=rng.standard_normal((E, h, d)) / np.sqrt(h))
    if request.param == "learned":
        inp["W_r"] = rng.standard_normal((d, E))
        inp["b"] = rng.standard_normal(E)
    else:
        inp["idx"] = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        inp["glogit"] = rng.standard_normal((T, k))
    dY = rng.standard_normal((T, d))
    return request.param, inp, dY, k, E


def test_backward_matches_finite_differences(tiny):
    routing, inp, dY, k, E = tiny
    fwd = ol.layer_forward(inp, k, E, logits_dtype=np.float64)
    bw = ol.layer_backward(dict(inp, dY=dY), fwd, k, E)
    for key, g in (("W1", bw["dW1"]), ("W3", bw["dW3"]), ("W2", bw["dW2"]),
                   ("x", bw["dX"])):
        _fd_check(inp, key, g, k, E, dY)
    if routing == "learned":
        _fd_check(inp, "W_r", bw["dW_r"], k, E, dY)
        _fd_check(inp, "b", bw["db"], k, E, dY)
    else:
        # gate logits: the gradient sits at the selected experts' columns of dz
        gl = np.take_along_axis(bw["dz"], inp["idx"].astype(np.int64), axis=1)
        _fd_check(inp, "glogit", gl, k, E, dY)


def test_empty_expert_weight_gradient_is_exactly_zero():
    T, d, E, k, h = 5, 8, 4, 2, 6
    rng = np.random.default_rng(12)
    idx = np.array([[0, 1], [1, 3], [3, 0], [0, 1], [1, 3]], np.int32)   # expert 2 empty
    inp = dict(x=rng.standard_normal((T, d)),
               W1=rng.standard_normal((E, d, h)), W3=rng.standard_normal((E, d, h)),
               W2=rng.standard_normal((E, h, d)), idx=idx,
               glogit=rng.standard_normal((T, k)), dY=rng.standard_normal((T, d)))
    fwd = ol.layer_forward(inp, k, E)
    bw = ol.layer_backward(inp, fwd, k, E)
    assert fwd["counts"][2] == 0
    for key in ("dW1", "dW3", "dW2"):
        assert np.all(bw[key][2] == 0.0)
        assert np.all(np.any(bw[key][[0, 1, 3]] != 0, axis=(1, 2)))


def test_identical_experts_gradients_sum_to_dense():
    # with identical experts, sum_e dW_e equals the dense FFN's weight gradient
    # for per-token upstream gradients g_j * dY (gates sum to 1 -> dY itself)
    T, d, E, k, h = 7, 6, 3, 2, 5
    rng = np.random.default_rng(13)
    W1 = np.broadcast_to(rng.standard_normal((d, h)), (E, d, h)).copy()
    W3 = np.broadcast_to(rng.standard_normal((d, h)), (E, d, h)).copy()
    W2 = np.broadcast_to(rng.standard_normal((h, d)), (E, h, d)).copy()
    inp = dict(x=rng.standard_normal((T, d)), W1=W1, W3=W3, W2=W2,
               idx=np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32),
               glogit=rng.standard_normal((T, k)), dY=rng.standard_normal((T, d)))
    fwd = ol.layer_forward(inp, k, E)
    bw = ol.layer_backward(inp, fwd, k, E)
    # dense single expert with all tokens, upstream gradient dY
    dense = dict(inp, W1=W1[:1], W3=W3[:1], W2=W2[:1],
                 idx=np.zeros((T, 1), np.int32), glogit=np.zeros((T, 1)))
    fd = ol.layer_forward(dense, 1, 1)
    bd = ol.layer_backward(dense, fd, 1, 1)
    for key in ("dW1", "dW3", "dW2"):
        np.testing.assert_allclose(bw[key].sum(0), bd[key][0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bw["dX"], bd["dX"], rtol=1e-10, atol=1e-12)
