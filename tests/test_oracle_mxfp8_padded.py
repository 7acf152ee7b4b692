"""Pins for the oracle's MXFP8 codec and the padded-capacity reference (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import layer as ol
from oracle import mxfp8 as mx
from oracle import padded as pd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_format.json")


def test_format_constants_from_the_pages():
    gold = json.load(open(GOLDEN))
    assert mx.E4M3_MAX == gold["e4m3_max"]
    assert mx.BLOCK == gold["block_elements"]
    # storage of one block: BLOCK E4M3 bytes + one E8M0 byte
    q, s = mx.quantize_blocks(np.ones((1, 4 * mx.BLOCK)))
    bits = 8 * (q.size + s.size) / q.size
    assert bits == gold["bits_per_element"]
    assert np.nanmax(mx.e4m3_decode(np.arange(256))) == gold["e4m3_max"]


def test_e4m3_decode_matches_library_on_all_codes():
    c = np.arange(256, dtype=np.uint8)
    ours = mx.e4m3_decode(c)
    lib = torch.from_numpy(c).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()
    assert np.isnan(ours[[0x7F, 0xFF]]).all() and np.isfinite(np.delete(ours, [0x7F, 0xFF])).all()


def test_e4m3_encode_roundtrip_and_library_rounding():
    c = np.arange(256)
    finite = ~np.isnan(mx.e4m3_decode(c))
    assert np.array_equal(mx.e4m3_encode(mx.e4m3_decode(c[finite])), c[finite])
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(50000) * 60, rng.standard_normal(50000) * 1e-2,
                        # exact midpoints between neighbouring codes (tie cases)
                        (mx.e4m3_decode(np.arange(1, 126)) + mx.e4m3_decode(np.arange(2, 127))) / 2])
    v = np.clip(v, -448, 448)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mx.e4m3_encode(v), lib)


def test_block_exponent_is_smallest_fitting_power():
    rng = np.random.default_rng(1)
    amax = np.concatenate([np.exp2(rng.uniform(-60, 60, 20000)),
                           448.0 * np.exp2(np.arange(-20, 20)),              # exact fits
                           np.nextafter(448.0 * np.exp2(np.arange(-20, 20)), np.inf)])
    e = mx.block_exponent(amax)
    assert np.all(amax <= 448.0 * np.exp2(e.astype(float)))
    assert np.all(amax > 448.0 * np.exp2(e.astype(float) - 1))
    assert mx.block_exponent(0.0) == -127


def test_qdq_error_bound():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-8, 8, (64, 1)))
    q, s = mx.quantize_blocks(v, axis=1)
    assert q.dtype == np.uint8 and s.shape == (64, 8)
    back = mx.dequantize_blocks(q, s, axis=1)
    e = (s.astype(float) - 127).repeat(32, axis=1)
    # half an E4M3 ulp: 2^-4 relative for normals, 2^-10 * 2^e absolute below
    bound = np.maximum(np.abs(v) * 2.0 ** -4, np.exp2(e - 10))
    assert np.all(np.abs(back - v) <= bound)
    # the scaled block maximum always fits: no code decodes above 448
    assert np.nanmax(np.abs(mx.e4m3_decode(q))) <= 448


def test_quantize_along_axis0_matches_transposed():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((64, 5))
    q0, s0 = mx.quantize_blocks(w, axis=0)
    q1, s1 = mx.quantize_blocks(w.T, axis=1)
    assert np.array_equal(q0, q1.T) and np.array_equal(s0, s1.T)


def test_padded_with_enough_capacity_equals_unpadded():
    T, d, E, k, h = 30, 8, 4, 2, 6
    rng = np.random.default_rng(4)
    inp = dict(x=rng.standard_normal((T, d)), W1=rng.standard_normal((E, d, h)),
               W3=rng.standard_normal((E, d, h)), W2=rng.standard_normal((E, h, d)),
               idx=np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32),
               glogit=rng.standard_normal((T, k)))
    ref = ol.layer_forward(inp, k, E)
    C = int(ref["counts"].max())
    p = pd.padded_forward(inp["x"], inp["idx"], ref["g"], inp["W1"], inp["W3"], inp["W2"], E, C)
    assert p["dropped"] == 0
    np.testing.assert_allclose(p["out"], ref["out"], rtol=1e-12, atol=1e-12)
    assert p["padded_rows"] == E * C and p["unpadded_rows"] == T * k


def test_padded_drops_overflow_by_hand():
    # T=4, k=1, E=2: expert 0 gets tokens 0,1,2 and expert 1 gets token 3.
    # Capacity 2 keeps tokens 0 and 1 at expert 0 and drops token 2.
    T, d, E, h = 4, 3, 2, 2
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, d, h)); W3 = rng.standard_normal((E, d, h))
    W2 = rng.standard_normal((E, h, d))
    idx = np.array([[0], [0], [0], [1]])
    assert pd.capacity(T, 1, E, factor=1.0) == 2
    assert pd.capacity(16384, 4, 128) == 640
    p = pd.padded_forward(x, idx, np.ones((T, 1)), W1, W3, W2, E, 2)
    assert p["dropped"] == 1 and p["dropped_fraction"] == 0.25
    assert list(p["kept"][:, 0]) == [True, True, False, True]
    assert np.all(p["out"][2] == 0)
    for t, e in ((0, 0), (1, 0), (3, 1)):
        ref = (ol.silu(x[t] @ W1[e]) * (x[t] @ W3[e])) @ W2[e]
        np.testing.assert_allclose(p["out"][t], ref, rtol=1e-12)


def test_qdq_is_exact_on_representable_blocks():
    # blocks whose values lie on the E4M3 grid times 2^s, with the block maximum
    # exactly 448 * 2^s, come back unchanged
    rng = np.random.default_rng(6)
    codes = rng.integers(0, 0x7E, (8, 4, 32))
    codes[:, :, 0] = 0x7E                                  # 448 in every block
    sgn = np.where(rng.random((8, 4, 32)) < 0.5, -1.0, 1.0)
    scale = np.exp2(rng.integers(-20, 20, (8, 4, 1)).astype(float))
    v = (sgn * mx.e4m3_decode(codes) * scale).reshape(8, 128)
    assert np.array_equal(mx.qdq(v, axis=1), v)


def test_mxfp8_forward_error_matches_format_precision():
    # E4M3 keeps 3 mantissa bits (about 2.6% RMS relative rounding per
    # operand); through two quantised GEMMs and a quantised activation the
    # output error of Gaussian data lands at a few percent, never at zero.
    T, d, E, k, h = 32, 128, 3, 2, 64
    rng = np.random.default_rng(7)
    Xp = rng.standard_normal((T * k, d))
    W1 = rng.standard_normal((E, d, h)) / np.sqrt(d); W3 = rng.standard_normal((E, d, h)) / np.sqrt(d)
    W2 = rng.standard_normal((E, h, d)) / np.sqrt(h)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    _, off, _, _ = ol.route_map(idx, E)
    exact = ol.expert_ffn_forward(Xp, off, W1, W3, W2)
    q = mx.expert_ffn_forward_mxfp8(Xp, off, W1, W3, W2)
    rel = np.linalg.norm(q["Yp"] - exact["Yp"]) / np.linalg.norm(exact["Yp"])
    assert 0.02 < rel < 0.12
    # the first GEMM alone: two quantised operands, ~3.7% expected
    h1 = mx.qdq(Xp, axis=1)[off[0]:off[1]] @ mx.qdq(W1[0], axis=0)
    h1x = Xp[off[0]:off[1]] @ W1[0]
    rel1 = np.linalg.norm(h1 - h1x) / np.linalg.norm(h1x)
    assert 0.015 < rel1 < 0.06


@pytest.mark.parametrize("case", ["Xp and W1/W3", "A and W2"])
def test_mxfp8_forward_blocks_run_along_each_reduction_dimension(case):
    # Powers of two from 2^-10 to 2^10 scale the rows of a GEMM's left operand
    # and the output columns of its right one.  A block of 32 along the
    # reduction dimension (the pages' rule) never holds two of those scales,
    # so once the column scales are divided out every output row keeps E4M3
    # precision; a block across rows or across output columns would span up
    # to 2^20, beyond E4M3's range of about 2^17.8, and flush or coarsen the
    # small members.  Case one checks H1, H3 (Xp, W1, W3); case two Yp (A, W2).
    T, d, E, k, h = 32, 64, 2, 2, 64
    R = T * k
    rng = np.random.default_rng(22 if case == "A and W2" else 21)
    p2 = lambda lo, hi, shape: np.exp2(rng.integers(lo, hi + 1, shape).astype(float))  # noqa: E731
    one = lambda n: np.ones((E, 1, n))  # noqa: E731
    if case == "Xp and W1/W3":
        sx, c1, c3, c2 = p2(-10, 10, (R, 1)), p2(-10, 10, (E, 1, h)), p2(-10, 10, (E, 1, h)), one(d)
        checks = (("H1", c1), ("H3", c3))
    else:                       # rows of A vary like those of Xp squared
        sx, c1, c3, c2 = p2(-5, 5, (R, 1)), one(h), one(h), p2(-10, 10, (E, 1, d))
        checks = (("Yp", c2),)
    Xp = rng.standard_normal((R, d)) * sx
    W1 = rng.standard_normal((E, d, h)) / 8 * c1
    W3 = rng.standard_normal((E, d, h)) / 8 * c3
    W2 = rng.standard_normal((E, h, d)) / 8 * c2
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    _, off, _, _ = ol.route_map(idx, E)
    with np.errstate(over="ignore"):        # silu of very negative inputs: exp overflows to -0
        exact = ol.expert_ffn_forward(Xp, off, W1, W3, W2)
        q = mx.expert_ffn_forward_mxfp8(Xp, off, W1, W3, W2)
    for name, cs in checks:
        rel = []
        for e in range(E):
            a = exact[name][off[e]:off[e + 1]] / cs[e]
            b = q[name][off[e]:off[e + 1]] / cs[e]
            rel.append(np.linalg.norm(b - a, axis=1) / np.linalg.norm(a, axis=1))
        rel = np.concatenate(rel)
        # two quantised operands: about 3.7 % a row; with A's as well about 6 %
        assert np.median(rel) < (0.06 if name != "Yp" else 0.12), (name, np.median(rel))
        assert rel.max() < (0.15 if name != "Yp" else 0.3), (name, rel.max())
        assert rel.min() > 0


def _padded_case(seed, T=12, d=5, E=3, k=2, h=4):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, d, h)) / 2; W3 = rng.standard_normal((E, d, h)) / 2
    W2 = rng.standard_normal((E, h, d)) / 2
    W_r = rng.standard_normal((d, E))
    dOut = rng.standard_normal((T, d))
    return x, W1, W3, W2, W_r, dOut


def test_padded_backward_finite_differences_with_drops():
    # learned router, capacity below the hottest expert's load: the central
    # differences of <dOut, out> must match every gradient the backward returns
    T, d, E, k, h = 12, 5, 3, 2, 4
    x, W1, W3, W2, W_r, dOut = _padded_case(11, T, d, E, k, h)
    idx = ol.topk(x @ W_r, k)
    C = 6
    counts = np.bincount(idx.reshape(-1), minlength=E)
    assert counts.max() > C                      # some slots are dropped

    def loss(x_, W1_, W3_, W2_, W_r_):
        g = ol.topk_gates(x_ @ W_r_, idx)
        return float((dOut * pd.padded_forward(x_, idx, g, W1_, W3_, W2_, E, C)["out"]).sum())

    g = ol.topk_gates(x @ W_r, idx)
    b = pd.padded_backward(x, idx, g, W1, W3, W2, dOut, E, C, W_r=W_r)
    args = [x, W1, W3, W2, W_r]
    eps = 1e-6
    for which, grad in ((0, b["dX"]), (1, b["dW1"]), (2, b["dW3"]), (3, b["dW2"]), (4, b["dW_r"])):
        num = np.zeros_like(args[which])
        for i in np.ndindex(args[which].shape):
            plus = [a.copy() for a in args]; minus = [a.copy() for a in args]
            plus[which][i] += eps; minus[which][i] -= eps
            num[i] = (loss(*plus) - loss(*minus)) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-5, atol=1e-6)
    # a dropped slot has no gate gradient; a kept one does
    p = pd.padded_forward(x, idx, g, W1, W3, W2, E, C)
    assert np.all(b["dg"][~p["kept"]] == 0) and np.all(b["dg"][p["kept"]] != 0)


def test_padded_backward_with_enough_capacity_equals_unpadded():
    T, d, E, k, h = 30, 8, 4, 2, 6
    rng = np.random.default_rng(12)
    inp = dict(x=rng.standard_normal((T, d)), W1=rng.standard_normal((E, d, h)),
               W3=rng.standard_normal((E, d, h)), W2=rng.standard_normal((E, h, d)),
               idx=np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32),
               glogit=rng.standard_normal((T, k)), dY=rng.standard_normal((T, d)))
    ref = ol.layer_forward(inp, k, E)
    refb = ol.layer_backward(inp, ref, k, E)
    C = int(ref["counts"].max()) + 3               # zero rows in every batch
    b = pd.padded_backward(inp["x"], inp["idx"], ref["g"], inp["W1"], inp["W3"], inp["W2"],
                           inp["dY"], E, C)
    for n, m in (("dX", "dX"), ("dg", "dg"), ("dW1", "dW1"), ("dW3", "dW3"), ("dW2", "dW2"),
                 ("dz", "dz")):
        np.testing.assert_allclose(b[n], refb[m], rtol=1e-11, atol=1e-11)


def test_padded_backward_drop_by_hand():
    # T=4, k=1, E=2, capacity 2: token 2 is dropped at expert 0, so it gets no
    # gradient, and expert 0's weight gradient comes from tokens 0 and 1 only
    T, d, E, h = 4, 3, 2, 2
    rng = np.random.default_rng(13)
    x = rng.standard_normal((T, d))
    W1 = rng.standard_normal((E, d, h)); W3 = rng.standard_normal((E, d, h))
    W2 = rng.standard_normal((E, h, d))
    dOut = rng.standard_normal((T, d))
    idx = np.array([[0], [0], [0], [1]])
    g = np.ones((T, 1))
    b = pd.padded_backward(x, idx, g, W1, W3, W2, dOut, E, 2)
    assert np.all(b["dX"][2] == 0) and b["dg"][2, 0] == 0
    kept = ol.expert_ffn_forward(x[:2], [0, 2], W1[:1], W3[:1], W2[:1])
    kb = ol.expert_ffn_backward(x[:2], [0, 2], W1[:1], W3[:1], W2[:1], kept["H1"], kept["H3"],
                                kept["A"], dOut[:2])
    for n in ("dW1", "dW3", "dW2"):
        np.testing.assert_allclose(b[n][0], kb[n][0], rtol=1e-12, atol=1e-12)


def test_capacity_route_map_by_hand_and_against_the_kept_mask():
    # T=4, k=1, E=2, C=2: expert 0 keeps tokens 0, 1 (rows 0, 1) and drops
    # token 2; expert 1 holds token 3 in row 2 and leaves row 3 empty
    idx = np.array([[0], [0], [0], [1]])
    c, o, ros, sor, routed = pd.capacity_route_map(idx, 2, 2)
    assert list(c) == [2, 1] and list(o) == [0, 2, 4] and list(routed) == [3, 1]
    assert list(ros) == [0, 1, -1, 2] and list(sor) == [0, 1, 3, -1]
    # larger: the kept slots are exactly padded_forward's, every kept row maps back
    T, d, E, k, h = 40, 4, 5, 3, 4
    rng = np.random.default_rng(14)
    idx = np.stack([rng.choice(E, k, replace=False, p=[.5, .2, .1, .1, .1]) for _ in range(T)])
    C = 18
    c, o, ros, sor, routed = pd.capacity_route_map(idx, E, C)
    x = rng.standard_normal((T, d))
    W = rng.standard_normal((E, d, h)); W2 = rng.standard_normal((E, h, d))
    p = pd.padded_forward(x, idx, np.ones((T, k)), W, W, W2, E, C)
    assert np.array_equal(ros >= 0, p["kept"].reshape(-1))
    assert np.array_equal(routed, np.bincount(idx.reshape(-1), minlength=E))
    kept = np.nonzero(ros >= 0)[0]
    assert np.array_equal(sor[ros[kept]], kept)
    assert (sor >= 0).sum() == kept.size == c.sum()
    for e in range(E):                           # kept rows fill the front of each block
        blk = sor[e * C:(e + 1) * C]
        assert np.all(blk[:c[e]] >= 0) and np.all(blk[c[e]:] == -1)
        assert np.all(np.diff(blk[:c[e]]) > 0)   # in slot order


def test_mxfp8_dgrad_exact_on_representable_operands_and_at_format_precision():
    # operands whose 32-blocks along h already lie on the E4M3 grid (block
    # maximum exactly 448 * 2^s) pass through the quantisation unchanged, so
    # the MXFP8 dgrad equals the exact expert dgrad; on Gaussian data its
    # error is set by E4M3's 3 mantissa bits (a few percent)
    rng = np.random.default_rng(15)
    T, d, E, k, h = 24, 64, 3, 2, 64

    def on_grid(shape):
        codes = rng.integers(0, 0x7E, shape + (h // 32, 32))
        codes[..., 0] = 0x7E
        sgn = np.where(rng.random(codes.shape) < 0.5, -1.0, 1.0)
        sc = np.exp2(rng.integers(-12, -4, shape + (h // 32, 1)).astype(float))
        return (sgn * mx.e4m3_decode(codes) * sc).reshape(shape + (h,))

    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    _, off, _, _ = ol.route_map(idx, E)
    dH1, dH3 = on_grid((T * k,)), on_grid((T * k,))
    W1 = np.stack([on_grid((d,)) for _ in range(E)]).transpose(0, 1, 2)    # [E, d, h]
    W3 = np.stack([on_grid((d,)) for _ in range(E)])
    exact = np.zeros((T * k, d))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        exact[lo:hi] = dH1[lo:hi] @ W1[e].T + dH3[lo:hi] @ W3[e].T
    got = mx.expert_dgrad_dx_mxfp8(dH1, dH3, off, W1, W3)
    np.testing.assert_allclose(got, exact, rtol=1e-12, atol=1e-12)
    # Gaussian operands: a few percent off the exact product, never zero
    dH1, dH3 = rng.standard_normal((T * k, h)), rng.standard_normal((T * k, h))
    W1, W3 = rng.standard_normal((E, d, h)), rng.standard_normal((E, d, h))
    exact = np.zeros((T * k, d))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        exact[lo:hi] = dH1[lo:hi] @ W1[e].T + dH3[lo:hi] @ W3[e].T
    got = mx.expert_dgrad_dx_mxfp8(dH1, dH3, off, W1, W3)
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert 0.015 < rel < 0.06
    # quantised along h: with weight rows whose magnitudes vary along d, every
    # output column stays at the format's precision, while quantising the
    # weights along d (the forward's axis) crushes the small rows of a block
    sc = np.exp2(rng.integers(-10, 11, (E, d, 1)).astype(float))   # one scale per output column
    W1, W3 = W1 * sc, W3 * sc
    exact = np.zeros((T * k, d)); wrong = np.zeros((T * k, d))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        exact[lo:hi] = dH1[lo:hi] @ W1[e].T + dH3[lo:hi] @ W3[e].T
        wrong[lo:hi] = (mx.qdq(dH1[lo:hi], axis=1) @ mx.qdq(W1[e], axis=0).T
                        + mx.qdq(dH3[lo:hi], axis=1) @ mx.qdq(W3[e], axis=0).T)
    got = mx.expert_dgrad_dx_mxfp8(dH1, dH3, off, W1, W3)
    def col_err(v):       # worst relative error of one expert's output column
        return max((np.linalg.norm(v[off[e]:off[e + 1]] - exact[off[e]:off[e + 1]], axis=0)
                    / np.linalg.norm(exact[off[e]:off[e + 1]], axis=0)).max()
                   for e in range(E) if off[e + 1] > off[e])
    assert col_err(got) < 0.1
    assert col_err(wrong) > 0.3
