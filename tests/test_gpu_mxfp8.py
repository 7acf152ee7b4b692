"""GPU parity of the MXFP8 path against the fp64 oracle.

Quantised codes and scales are compared bit-exactly (the inputs are bf16, so
the scaled value v * 2^-e is exact on both sides and RNE to E4M3 is one
function).  The block-scaled forward is compared with the oracle's
quantise -> dequantise -> exact-arithmetic mode within relative L2 4e-2; the
quantised activation A is computed on the device from fp32 accumulators, so
its codes are compared through their dequantised values."""
import numpy as np
import pytest
import torch

import oracle.layer as ol
import oracle.mxfp8 as om
from token_dispatch_grouped_router_gb300 import libmoe as L
from token_dispatch_grouped_router_gb300 import workloads as wl
from token_dispatch_grouped_router_gb300.layer import bf16_tensor

from gpu_helpers import assert_close, as_f64, ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"
MX_REL_L2 = 4e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    L.load()


def u8(t):
    return t.detach().cpu().numpy()


def _edge_values(rng, rows, K):
    v = rng.standard_normal((rows, K)).astype(np.float32)
    v[0] = 0.0                                              # all-zero block row
    v[1, :32] = np.float32(448.0) * np.float32(2.0) ** rng.integers(-20, 20)   # exact fits
    v[2] *= np.float32(1e-30)                               # tiny magnitudes
    v[3, ::2] = -0.0                                        # signed zeros
    v[4] *= np.float32(1e30)                                # huge magnitudes
    return wl.bf16_bits(v)


@pytest.mark.parametrize("rows,K", [(1, 32), (37, 96), (513, 2048)])
def test_quantize_rows_bit_exact(rows, K):
    rng = np.random.default_rng(rows + K)
    x = _edge_values(rng, max(rows, 5), K)[:rows]
    q = torch.empty(rows, K, dtype=torch.uint8, device=DEV)
    s = torch.empty(rows, K // 32, dtype=torch.uint8, device=DEV)
    L.moe_mxfp8_quantize_rows(bf16_tensor(x, DEV), q, s)
    qr, sr = om.quantize_blocks(x, axis=1)
    assert np.array_equal(u8(s), sr)
    assert np.array_equal(u8(q), qr)


@pytest.mark.parametrize("E,K,N", [(2, 64, 128), (3, 256, 384), (8, 2048, 1024)])
def test_quantize_weights_bit_exact(E, K, N):
    rng = np.random.default_rng(E * K)
    W = wl.bf16_bits(rng.standard_normal((E, K, N)).astype(np.float32) / np.sqrt(K))
    wq = torch.empty(E, N, K, dtype=torch.uint8, device=DEV)
    ws = torch.empty(E, N, K // 32, dtype=torch.uint8, device=DEV)
    L.moe_mxfp8_quantize_weights(bf16_tensor(W, DEV), wq, ws)
    gq, gs = u8(wq), u8(ws)
    for e in range(E):
        qr, sr = om.quantize_blocks(W[e], axis=0)           # blocks along K for every column
        assert np.array_equal(gs[e], sr.T), e
        assert np.array_equal(gq[e], qr.T), e


@pytest.mark.parametrize("E,K,N", [(2, 64, 128), (3, 256, 384), (8, 2048, 1024)])
def test_quantize_weights_from_fp32_masters_bit_exact(E, K, N):
    # fp32 masters carry bits below bf16's mantissa: one rounding to E4M3
    rng = np.random.default_rng(E * K + 1)
    W = (rng.standard_normal((E, K, N)) / np.sqrt(K)).astype(np.float32)
    W[0, :32, 0] = 0.0                                      # an all-zero block
    W[0, :32, 1] = np.float32(448.0) * np.float32(2.0) ** -7  # a block max that fits exactly
    W[-1, -32:, -1] *= np.float32(1e-35)                    # fp32 subnormals and tiny values
    W[-1, -32:, -2] *= np.float32(1e30)
    wq = torch.empty(E, N, K, dtype=torch.uint8, device=DEV)
    ws = torch.empty(E, N, K // 32, dtype=torch.uint8, device=DEV)
    L.moe_mxfp8_quantize_weights_f32(torch.from_numpy(W).to(DEV), wq, ws)
    gq, gs = u8(wq), u8(ws)
    for e in range(E):
        qr, sr = om.quantize_blocks(W[e].astype(np.float64), axis=0)
        assert np.array_equal(gs[e], sr.T), e
        assert np.array_equal(gq[e], qr.T), e


def _atoms_of(scales, cols, K, second=None):
    """Expected atom bytes of row-major scales [E][N][K/32] for column tiles of
    `cols` (96: rows of `scales` then the same rows of `second`; 192: rows of
    `scales`): per (expert, tile, 128-deep k-block) two 512-byte atoms, byte
    (c % 32) * 16 + ((c % 128) // 32) * 4 + q of atom c // 128 = the scale of
    tile column c for 32-block q of the k-block."""
    E, N, _ = scales.shape
    KB = K // 128
    NT = -(-N // cols)
    out = np.zeros((E, NT, KB, 2, 32, 4, 4), np.uint8)   # [..][atom][r][j][q]
    for c in range(192):
        for nt in range(NT):
            if cols == 96:
                tab, n = (scales, nt * 96 + c) if c < 96 else (second, nt * 96 + c - 96)
            else:
                tab, n = scales, nt * 192 + c
            if n >= N:
                continue
            blk = tab[:, n, :].reshape(E, KB, 4)             # [e][kb][q]
            out[:, nt, :, c // 128, c % 32, (c % 128) // 32, :] = blk
    return out.reshape(-1)


@pytest.mark.parametrize("E,d,h", [(2, 128, 128), (3, 256, 384), (2, 512, 256)])
def test_weight_scale_atoms_layout(E, d, h):
    # the GEMM's atom order of the weight scales, byte for byte
    rng = np.random.default_rng(E + d + h)
    w1s = rng.integers(0, 255, (E, h, d // 32), dtype=np.uint8)
    w3s = rng.integers(0, 255, (E, h, d // 32), dtype=np.uint8)
    w2s = rng.integers(0, 255, (E, d, h // 32), dtype=np.uint8)
    n = L.moe_mxfp8_weight_atom_bytes(E, d, h)
    atoms = torch.full((n,), 7, dtype=torch.uint8, device=DEV)
    L.moe_mxfp8_weight_scale_atoms(*(torch.from_numpy(a).to(DEV) for a in (w1s, w3s, w2s)), atoms)
    up = _atoms_of(w1s, 96, d, second=w3s)
    dn = _atoms_of(w2s, 192, h)
    assert n == up.size + dn.size
    got = u8(atoms)
    assert np.array_equal(got[:up.size], up)
    assert np.array_equal(got[up.size:], dn)


@pytest.mark.parametrize("rows,K", [(1, 32), (37, 96), (513, 2048)])
def test_dequantize_rows_bit_exact(rows, K):
    # codes and scales from the oracle's quantiser, including tiny and huge
    # scales; the device value code * 2^(s-127) rounded to bf16 must equal the
    # oracle's exact value rounded to bf16 (RNE, by torch)
    rng = np.random.default_rng(rows * K)
    x = _edge_values(rng, max(rows, 5), K)[:rows]
    qr, sr = om.quantize_blocks(x, axis=1)
    q = torch.from_numpy(qr).to(DEV)
    s = torch.from_numpy(np.ascontiguousarray(sr)).to(DEV)
    out = torch.empty(rows, K, dtype=torch.bfloat16, device=DEV)
    L.moe_mxfp8_dequantize_rows(q, s, out)
    exact = om.dequantize_blocks(qr, sr, axis=1)
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), exact)   # exact in fp32
    ref = torch.from_numpy(exact.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(out.cpu().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("T,d,k", [(5, 32, 1), (300, 2048, 4), (77, 96, 2)])
def test_dispatch_mxfp8_bit_exact(T, d, k):
    E = 8
    rng = np.random.default_rng(T + d)
    x = _edge_values(rng, T, d) if T >= 5 else wl.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    _, _, ros, _ = ol.route_map(idx, E)
    xq = torch.empty(T * k, d, dtype=torch.uint8, device=DEV)
    xs = torch.empty(T * k, d // 32, dtype=torch.uint8, device=DEV)
    xp = torch.empty(T * k, d, dtype=torch.bfloat16, device=DEV)
    L.moe_dispatch_rows_mxfp8(bf16_tensor(x, DEV), torch.from_numpy(ros).to(DEV), k, xq, xs, xp)
    qr, sr = om.quantize_blocks(x, axis=1)
    slots = np.arange(T * k)
    assert np.array_equal(u8(xq)[ros[slots]], qr[slots // k])
    assert np.array_equal(u8(xs)[ros[slots]], sr[slots // k])
    assert np.array_equal(as_f64(xp), ol.dispatch(x, ros, k))


def _mx_layer(w, inp):
    """Device MXFP8 forward of workload w: weight quantisation, route map,
    quantising dispatch, block-scaled grouped GEMMs."""
    T, d, E, k, h = w.T, w.d, w.E, w.k, w.h
    R = T * k
    dev = DEV
    t = {}
    for n in ("W1", "W3", "W2"):
        t[n] = bf16_tensor(inp[n], dev)
    u = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)  # noqa: E731
    b = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)  # noqa: E731
    t["w1q"], t["w1s"] = u(E, h, d), u(E, h, d // 32)
    t["w3q"], t["w3s"] = u(E, h, d), u(E, h, d // 32)
    t["w2q"], t["w2s"] = u(E, d, h), u(E, d, h // 32)
    L.moe_mxfp8_quantize_weights(t["W1"], t["w1q"], t["w1s"])
    L.moe_mxfp8_quantize_weights(t["W3"], t["w3q"], t["w3s"])
    L.moe_mxfp8_quantize_weights(t["W2"], t["w2q"], t["w2s"])
    t["w_atoms"] = u(L.moe_mxfp8_weight_atom_bytes(E, d, h))
    L.moe_mxfp8_weight_scale_atoms(t["w1s"], t["w3s"], t["w2s"], t["w_atoms"])
    idx = torch.from_numpy(np.ascontiguousarray(inp["idx"])).to(dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ros = torch.empty(R, dtype=torch.int32, device=dev)
    sor = torch.empty(R, dtype=torch.int32, device=dev)
    ws = torch.zeros(L.moe_workspace_size(T, E, k, d, h), dtype=torch.uint8, device=dev)
    L.moe_expert_offsets(idx, E, counts, offs, ros, sor, ws)
    t["xq"], t["xs"], t["xp"] = u(R, d), u(R, d // 32), b(R, d)
    L.moe_dispatch_rows_mxfp8(bf16_tensor(inp["x"], dev), ros, k, t["xq"], t["xs"], t["xp"])
    t["h1"], t["h3"], t["a"], t["yp"] = b(R, h), b(R, h), b(R, h), b(R, d)
    t["aq"], t["as"] = u(R, h), u(R, h // 32)
    L.moe_reset_status(ws)
    L.moe_grouped_swiglu_fwd_mxfp8(t["xq"], t["xs"], offs, t["w1q"], t["w3q"], t["w2q"],
                                   t["w_atoms"], t["h1"], t["h3"], t["a"], t["aq"], t["as"],
                                   t["yp"], ws)
    torch.cuda.synchronize()
    assert L.moe_get_status(ws) == 0
    t["offsets"] = offs
    t["ros"] = ros
    return t


@pytest.mark.parametrize("T,d,E,k,h,empty", [
    (300, 256, 6, 2, 384, (2,)),       # ragged rows, three 128-column blocks of h
    (1000, 512, 16, 4, 256, (0, 15)),
    (64, 128, 1, 1, 128, ()),
    # several 128-row tiles per expert, ragged tails
    (1500, 256, 2, 1, 384, ()),
    (2600, 512, 4, 2, 256, (1,)),
    (700, 128, 1, 1, 128, ()),
    # CTA pairs whose last 256-row tile leaves the odd CTA without rows
    (1100, 128, 1, 1, 128, ()),
    # CTA pairs, experts whose rows start off a 128-row boundary, d not a
    # multiple of the 192-column tile
    (3100, 640, 3, 2, 384, ()),
])
def test_grouped_forward_mxfp8_small(T, d, E, k, h, empty, record_property):
    w = wl.small_workload(T=T, d=d, E=E, k=k, h=h)
    inp = wl.generate(w, seed=2, with_backward=False)
    if empty:
        keep = [e for e in range(E) if e not in empty]
        rng = np.random.default_rng(3)
        inp["idx"] = np.stack([rng.permutation(keep)[:k] for _ in range(T)]).astype(np.int32)
    t = _mx_layer(w, inp)
    c, off, ros, _ = ol.route_map(inp["idx"], E)
    Xp = ol.dispatch(inp["x"], ros, k)
    ref = om.expert_ffn_forward_mxfp8(Xp, off, inp["W1"], inp["W3"], inp["W2"])
    assert_close(t["h1"], ref["H1"], "h1")
    assert_close(t["h3"], ref["H3"], "h3")
    assert_close(t["a"], ref["A"], "a")
    # device-quantised a, dequantised, against the exact a it came from
    aq_dq = om.dequantize_blocks(u8(t["aq"]), u8(t["as"]), axis=1)
    assert_close(aq_dq, ref["A"], "a quantised", rel_l2=MX_REL_L2, max_abs=0.1)
    assert_close(t["yp"], ref["Yp"], "yp", rel_l2=MX_REL_L2, max_abs=0.1)
    exact = ol.expert_ffn_forward(Xp, off, inp["W1"], inp["W3"], inp["W2"])["Yp"]
    rel = np.linalg.norm(as_f64(t["yp"]) - exact) / np.linalg.norm(exact)
    # the MXFP8 output against the unquantised fp64 layer: reported (pytest -s
    # prints it; junit XML carries it as a property) and bounded by what E4M3's
    # 3 mantissa bits allow through two quantised GEMMs and a quantised A
    rel_q = np.linalg.norm(as_f64(t["yp"]) - ref["Yp"]) / np.linalg.norm(ref["Yp"])
    record_property("yp_rel_l2_vs_unquantised", float(rel))
    record_property("yp_rel_l2_vs_quantised", float(rel_q))
    print(f"\nMXFP8 yp T={T} d={d} E={E} k={k} h={h}: rel-L2 {rel:.4f} vs the unquantised "
          f"layer, {rel_q:.2e} vs the quantise-dequantise oracle")
    assert 0.02 < rel < 0.12
    for e in empty:
        assert c[e] == 0


def test_full_size_mxfp8_sampled():
    w = wl.get_workload("train_e128")
    inp = wl.generate(w, seed=0, with_backward=False)
    t = _mx_layer(w, inp)
    k = w.k
    c, off, ros, sor = ol.route_map(inp["idx"], w.E)
    assert np.array_equal(t["offsets"].cpu().numpy(), off)
    rng = np.random.default_rng(11)
    toks = np.sort(rng.choice(w.T, 12, replace=False))
    rows, yref, href = [], [], []
    x = inp["x"]
    for tk in toks:
        for j in range(k):
            e = int(inp["idx"][tk, j])
            Xq = om.qdq(ol.decode_bf16(x[tk:tk + 1]), axis=1)
            w1 = om.qdq(inp["W1"][e], axis=0); w3 = om.qdq(inp["W3"][e], axis=0)
            w2 = om.qdq(inp["W2"][e], axis=0)
            H1 = Xq @ w1
            A = ol.silu(H1) * (Xq @ w3)
            yref.append((om.qdq(A, axis=1) @ w2)[0]); href.append(H1[0])
            rows.append(int(ros[tk * k + j]))
    rt = torch.tensor(rows, device=DEV, dtype=torch.long)
    assert_close(t["h1"][rt], np.array(href), "h1")
    assert_close(t["yp"][rt], np.array(yref), "yp", rel_l2=MX_REL_L2, max_abs=0.1)


def test_layer_step_mxfp8_forward_bf16_backward():
    # the layer's MXFP8 step: forward through the block-scaled GEMMs, backward
    # in bf16 from the forward's stored activations; the oracle composes its
    # quantise->dequantise forward with the analytic backward at those values
    from token_dispatch_grouped_router_gb300.layer import MoELayer
    w = wl.small_workload(T=500, d=256, E=8, k=2, h=256)
    inp = wl.generate(w, seed=5)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=False, device=DEV)
    layer.load_inputs(inp)
    layer.enable_mxfp8()
    L.moe_reset_status(layer.ws)
    layer.step_mxfp8()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    k, E = w.k, w.E
    g = ol.softmax_gates(inp["glogit"])
    _, off, ros, _ = ol.route_map(inp["idx"], E)
    Xp = ol.dispatch(inp["x"], ros, k)
    f = om.expert_ffn_forward_mxfp8(Xp, off, inp["W1"], inp["W3"], inp["W2"])
    assert_close(layer.out, ol.combine(f["Yp"], ros, g, k), "out", rel_l2=MX_REL_L2, max_abs=0.1)
    dYp, dg = ol.combine_backward(inp["dY"], f["Yp"], ros, g, k)
    b = ol.expert_ffn_backward(Xp, off, inp["W1"], inp["W3"], inp["W2"], f["H1"], f["H3"], f["A"], dYp)
    for n, key in (("dxp", "dXp"), ("dW1", "dW1"), ("dW3", "dW3"), ("dW2", "dW2")):
        assert_close(getattr(layer, n), b[key], n, rel_l2=MX_REL_L2, max_abs=0.1)
    assert_close(layer.dgate, dg, "dgate", rel_l2=MX_REL_L2, max_abs=0.1)


@pytest.mark.parametrize("T,E,k", [(500, 8, 2), (2600, 4, 2)])   # 128-row tiles / several per expert
def test_layer_step_mxfp8_saved_activations(T, E, k):
    # the MXFP8 step that keeps Xp and A only as codes + scales: the forward
    # writes no bf16 copy of either, the backward reads them back dequantised.
    # The oracle composes its quantise->dequantise forward with the analytic
    # backward at the dequantised Xp and A.
    from token_dispatch_grouped_router_gb300.layer import MoELayer
    w = wl.small_workload(T=T, d=256, E=E, k=k, h=256)
    inp = wl.generate(w, seed=6)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=False, device=DEV)
    layer.load_inputs(inp)
    layer.enable_mxfp8()
    layer.xp.fill_(float("nan")); layer.a.fill_(float("nan"))     # nothing may read stale copies
    L.moe_reset_status(layer.ws)
    layer.quantize_weights()
    layer.forward_mxfp8(saved="mxfp8")
    torch.cuda.synchronize()
    assert torch.isnan(layer.xp.float()).all() and torch.isnan(layer.a.float()).all()
    layer.restore_saved_mxfp8()
    layer.backward()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    g = ol.softmax_gates(inp["glogit"])
    _, off, ros, _ = ol.route_map(inp["idx"], E)
    Xp = ol.dispatch(inp["x"], ros, k)
    f = om.expert_ffn_forward_mxfp8(Xp, off, inp["W1"], inp["W3"], inp["W2"])
    Xq = om.qdq(Xp, axis=1)
    # the dequantised rows are exactly the oracle's quantise->dequantise rows
    assert np.array_equal(as_f64(layer.xp), Xq)
    Aq = om.qdq(f["A"], axis=1)
    assert_close(layer.a, Aq, "a (dequantised)", rel_l2=MX_REL_L2, max_abs=0.1)
    assert_close(layer.out, ol.combine(f["Yp"], ros, g, k), "out", rel_l2=MX_REL_L2, max_abs=0.1)
    dYp, dg = ol.combine_backward(inp["dY"], f["Yp"], ros, g, k)
    b = ol.expert_ffn_backward(Xq, off, inp["W1"], inp["W3"], inp["W2"], f["H1"], f["H3"], Aq, dYp)
    for n, key in (("dxp", "dXp"), ("dW1", "dW1"), ("dW3", "dW3"), ("dW2", "dW2")):
        assert_close(getattr(layer, n), b[key], n, rel_l2=MX_REL_L2, max_abs=0.1)
    assert_close(layer.dgate, dg, "dgate", rel_l2=MX_REL_L2, max_abs=0.1)


# ------------------------------------------------------------ MXFP8 dgrad

def test_dx_weight_scale_atoms_layout():
    # the dgrad GEMM's atoms: 192-column tiles of d, k-blocks of K = 2h with
    # W1's scales first, then W3's
    E, d, h = 2, 640, 256
    rng = np.random.default_rng(21)
    w1s = rng.integers(0, 255, (E, d, h // 32), dtype=np.uint8)
    w3s = rng.integers(0, 255, (E, d, h // 32), dtype=np.uint8)
    n = L.moe_mxfp8_dx_weight_atom_bytes(E, d, h)
    atoms = torch.full((n,), 7, dtype=torch.uint8, device=DEV)
    L.moe_mxfp8_dx_weight_scale_atoms(torch.from_numpy(w1s).to(DEV), torch.from_numpy(w3s).to(DEV), atoms)
    both = np.concatenate([w1s, w3s], axis=2)               # [E][d][2h/32]: K = 2h
    ref = _atoms_of(both, 192, 2 * h)
    assert n == ref.size
    assert np.array_equal(u8(atoms), ref)


def _dx_inputs(T, d, E, k, h, seed, empty=()):
    rng = np.random.default_rng(seed)
    keep = [e for e in range(E) if e not in empty]
    idx = np.stack([rng.permutation(keep)[:k] for _ in range(T)]).astype(np.int32)
    _, off, _, _ = ol.route_map(idx, E)
    R = T * k
    dh1 = wl.bf16_bits((rng.standard_normal((R, h)) * 0.1).astype(np.float32))
    dh3 = wl.bf16_bits((rng.standard_normal((R, h)) * 0.1).astype(np.float32))
    W1 = wl.bf16_bits((rng.standard_normal((E, d, h)) / np.sqrt(d)).astype(np.float32))
    W3 = wl.bf16_bits((rng.standard_normal((E, d, h)) / np.sqrt(d)).astype(np.float32))
    return off, dh1, dh3, W1, W3


def _device_dx_mxfp8(off, dh1, dh3, W1, W3, E, d, h):
    R = dh1.shape[0]
    u = lambda *s: torch.empty(s, dtype=torch.uint8, device=DEV)  # noqa: E731
    t = {}
    for n, v in (("dh1", dh1), ("dh3", dh3)):
        t[n + "q"], t[n + "s"] = u(R, h), u(R, h // 32)
        L.moe_mxfp8_quantize_rows(bf16_tensor(v, DEV), t[n + "q"], t[n + "s"])
    for n, v in (("w1", W1), ("w3", W3)):
        t[n + "q"], t[n + "s"] = u(E, d, h), u(E, d, h // 32)
        L.moe_mxfp8_quantize_rows(bf16_tensor(v, DEV).view(E * d, h), t[n + "q"].view(E * d, h),
                                  t[n + "s"].view(E * d, h // 32))
    atoms = u(L.moe_mxfp8_dx_weight_atom_bytes(E, d, h))
    L.moe_mxfp8_dx_weight_scale_atoms(t["w1s"], t["w3s"], atoms)
    dxp = torch.full((R, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(L.moe_workspace_size(R, E, 1, d, h), dtype=torch.uint8, device=DEV)
    L.moe_reset_status(ws)
    L.moe_grouped_swiglu_bwd_dx_mxfp8(t["dh1q"], t["dh1s"], t["dh3q"], t["dh3s"],
                                      torch.from_numpy(off.astype(np.int32)).to(DEV), t["w1q"], t["w3q"],
                                      atoms, dxp, ws)
    torch.cuda.synchronize()
    assert L.moe_get_status(ws) == 0
    return dxp


@pytest.mark.parametrize("T,d,E,k,h,empty", [
    (300, 256, 6, 2, 384, (2,)),       # single CTAs, ragged rows, an empty expert
    (1000, 640, 16, 4, 256, ()),       # d not a multiple of the 192-column tile
    (2600, 512, 4, 2, 256, (1,)),      # CTA pairs
    (1100, 128, 1, 1, 128, ()),        # CTA pairs, the odd CTA of the last tile without rows
])
def test_dgrad_mxfp8_small(T, d, E, k, h, empty, record_property):
    off, dh1, dh3, W1, W3 = _dx_inputs(T, d, E, k, h, seed=T + d, empty=empty)
    dxp = _device_dx_mxfp8(off, dh1, dh3, W1, W3, E, d, h)
    dec = ol.decode_bf16
    ref = om.expert_dgrad_dx_mxfp8(dec(dh1), dec(dh3), off, dec(W1), dec(W3))
    assert_close(dxp, ref, "dxp", rel_l2=MX_REL_L2, max_abs=0.1)
    exact = np.zeros_like(ref)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        exact[lo:hi] = dec(dh1)[lo:hi] @ dec(W1)[e].T + dec(dh3)[lo:hi] @ dec(W3)[e].T
    rel_q = np.linalg.norm(as_f64(dxp) - ref) / np.linalg.norm(ref)
    rel = np.linalg.norm(as_f64(dxp) - exact) / np.linalg.norm(exact)
    record_property("dxp_rel_l2_vs_quantised", float(rel_q))
    record_property("dxp_rel_l2_vs_unquantised", float(rel))
    print(f"\nMXFP8 dxp T={T} d={d} E={E} k={k} h={h}: rel-L2 {rel_q:.2e} vs the quantise-dequantise "
          f"oracle, {rel:.4f} vs the unquantised product")
    assert rel_q < 1e-2 and 0.01 < rel < 0.08


def test_layer_step_mxfp8_dgrad():
    # the layer step with the forward GEMMs and the dgrad GEMM in MXFP8: the
    # oracle composes its quantise->dequantise forward, the analytic backward
    # at those values and its MXFP8 dgrad of the rows
    from token_dispatch_grouped_router_gb300.layer import MoELayer
    w = wl.small_workload(T=2600, d=256, E=4, k=2, h=256)
    inp = wl.generate(w, seed=9)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=False, device=DEV)
    layer.load_inputs(inp)
    layer.enable_mxfp8()
    L.moe_reset_status(layer.ws)
    layer.step_mxfp8(dgrad="mxfp8")
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    k, E = w.k, w.E
    g = ol.softmax_gates(inp["glogit"])
    _, off, ros, _ = ol.route_map(inp["idx"], E)
    Xp = ol.dispatch(inp["x"], ros, k)
    f = om.expert_ffn_forward_mxfp8(Xp, off, inp["W1"], inp["W3"], inp["W2"])
    dYp, dg = ol.combine_backward(inp["dY"], f["Yp"], ros, g, k)
    b = ol.expert_ffn_backward(Xp, off, inp["W1"], inp["W3"], inp["W2"], f["H1"], f["H3"], f["A"], dYp)
    dXp = om.expert_dgrad_dx_mxfp8(b["dH1"], b["dH3"], off, ol.decode_bf16(inp["W1"]),
                                   ol.decode_bf16(inp["W3"]))
    for n, ref in (("dh1", b["dH1"]), ("dh3", b["dH3"]), ("dxp", dXp),
                   ("dX", ol.unpermute_sum(dXp, ros, k)), ("dW1", b["dW1"]), ("dW2", b["dW2"])):
        assert_close(getattr(layer, n), ref, n, rel_l2=MX_REL_L2, max_abs=0.1)


def test_full_size_dgrad_mxfp8_sampled():
    # train_e128 sizes (T = 32768, d = 2048, h = 1024, E = 128, top-4): the
    # layer's MXFP8 dgrad rows against the oracle's, from the device's dh1/dh3
    from token_dispatch_grouped_router_gb300.layer import MoELayer
    w = wl.get_workload("train_e128")
    inp = wl.generate(w, seed=0)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=False, device=DEV)
    layer.load_inputs(inp)
    layer.enable_mxfp8()
    L.moe_reset_status(layer.ws)
    layer.step_mxfp8(dgrad="mxfp8")
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    off = layer.offsets.cpu().numpy().astype(np.int64)
    rng = np.random.default_rng(13)
    experts = sorted(set(int(e) for e in rng.choice(w.E, 3, replace=False)))
    rows, ref = [], []
    dh1 = as_f64(layer.dh1); dh3 = as_f64(layer.dh3)
    for e in experts:
        rr = np.sort(rng.choice(np.arange(off[e], off[e + 1]), 4, replace=False))
        w1 = om.qdq(ol.decode_bf16(inp["W1"][e]), axis=1); w3 = om.qdq(ol.decode_bf16(inp["W3"][e]), axis=1)
        ref.append(om.qdq(dh1[rr], axis=1) @ w1.T + om.qdq(dh3[rr], axis=1) @ w3.T)
        rows.extend(rr.tolist())
    got = layer.dxp[torch.tensor(rows, device=DEV, dtype=torch.long)]
    assert_close(got, np.concatenate(ref), "dxp", rel_l2=MX_REL_L2, max_abs=0.1)


def test_mxfp8_step_captures_into_a_graph():
    # the MXFP8 step (forward and dgrad block-scaled, weights re-quantised in
    # the step) has no host synchronisation either: captured and replayed, it
    # reproduces the eager step bit for bit
    from token_dispatch_grouped_router_gb300.layer import MoELayer
    w = wl.small_workload(T=1300, d=256, E=4, k=2, h=256)
    inp = wl.generate(w, seed=12)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=False, device=DEV)
    layer.load_inputs(inp)
    layer.enable_mxfp8()
    step = lambda: layer.step_mxfp8(requantize=True, dgrad="mxfp8")  # noqa: E731
    step()
    torch.cuda.synchronize()
    names = ("out", "dxp", "dX", "dW1", "dW2", "dgate", "aq")
    eager = {n: getattr(layer, n).clone() for n in names}
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    for n in ("out", "dxp", "dX", "dW1", "dW2"):
        getattr(layer, n).zero_()
    g.replay()
    torch.cuda.synchronize()
    for n, v in eager.items():
        assert torch.equal(getattr(layer, n), v), n


@pytest.mark.parametrize("T,E,k", [(500, 8, 2), (2600, 4, 2)])   # single CTAs / CTA pairs
def test_dact_with_quantised_outputs(T, E, k):
    # the dact epilogue also writing dh1 / dh3 quantised along h: the bf16
    # outputs are those of the plain call bit for bit, and the codes and scales
    # are the oracle's MXFP8 blocks of those bf16 values, bit for bit
    from token_dispatch_grouped_router_gb300.layer import MoELayer
    w = wl.small_workload(T=T, d=256, E=E, k=k, h=384)
    inp = wl.generate(w, seed=16)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=False, device=DEV)
    layer.load_inputs(inp)
    layer.step()
    torch.cuda.synchronize()
    R, h = layer.R, w.h
    dh1 = torch.empty_like(layer.dh1); dh3 = torch.empty_like(layer.dh3)
    u = lambda *s: torch.full(s, 0xEE, dtype=torch.uint8, device=DEV)  # noqa: E731
    q1, s1, q3, s3 = u(R, h), u(R, h // 32), u(R, h), u(R, h // 32)
    L.moe_reset_status(layer.ws)
    L.moe_grouped_swiglu_bwd_dact_mxfp8(layer.offsets, layer.W2, layer.h1, layer.h3, layer.dyp,
                                        dh1, dh3, q1, s1, q3, s3, layer.ws)
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    assert torch.equal(dh1, layer.dh1) and torch.equal(dh3, layer.dh3)
    for q, sc, src in ((q1, s1, dh1), (q3, s3, dh3)):
        rq, rs = om.quantize_blocks(as_f64(src), axis=1)
        assert np.array_equal(u8(q), rq) and np.array_equal(u8(sc), rs)
