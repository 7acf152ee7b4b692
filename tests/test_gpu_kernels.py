"""GPU parity of the router, route-map and row-permute kernels against the
fp64 oracle, called through the C ABI (bit-exact for integer outputs)."""
import numpy as np
import pytest
import torch

import oracle.layer as ol
from token_dispatch_grouped_router_gb300 import libmoe as L
from token_dispatch_grouped_router_gb300 import workloads as wl
from token_dispatch_grouped_router_gb300.layer import bf16_tensor

from gpu_helpers import assert_close, as_f64, ensure_built, i32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    L.load()


def _ws(T, E, k, d=64, h=64):
    return torch.zeros(L.moe_workspace_size(T, E, k, d, h), dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (37, 8, 2), (515, 33, 4), (256, 128, 8),
                                   (64, 1024, 4), (300, 200, 8), (1000, 64, 1)])
def test_topk_bit_exact_with_ties(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    z = rng.standard_normal((T, E)).astype(np.float32)
    # force exact ties and signed zeros in a quarter of the rows
    z[::4] = rng.choice(np.array([-1.0, -0.0, 0.0, 0.5], np.float32), size=z[::4].shape)
    zt = torch.from_numpy(z).to(DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    g = torch.empty(T, k, dtype=torch.float32, device=DEV)
    L.moe_router_topk(zt, k, idx, g)
    ref = ol.topk(z, k)
    assert np.array_equal(i32(idx), ref)
    assert_close(g, ol.topk_gates(z, ref), "gates", rel_l2=1e-6, max_abs=1e-6)
    np.testing.assert_allclose(as_f64(g).sum(1), 1.0, atol=1e-6)


def test_router_gates_and_topk_backward():
    T, E, k = 777, 96, 4
    rng = np.random.default_rng(1)
    sel = rng.standard_normal((T, k)).astype(np.float32)
    g = torch.empty(T, k, dtype=torch.float32, device=DEV)
    L.moe_router_gates(torch.from_numpy(sel).to(DEV), g)
    gref = ol.softmax_gates(sel)
    assert_close(g, gref, "gates", rel_l2=1e-6, max_abs=1e-6)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    dg = rng.standard_normal((T, k)).astype(np.float32)
    dz = torch.full((T, E), 7.0, dtype=torch.float32, device=DEV)
    L.moe_router_topk_bwd(g, torch.from_numpy(dg).to(DEV), torch.from_numpy(idx).to(DEV), E, dz)
    ref = ol.router_topk_backward(as_f64(g), dg, idx, E)
    assert_close(dz, ref, "dlogits", rel_l2=1e-5, max_abs=1e-5)
    assert np.all(as_f64(dz)[ref == 0] == 0)


@pytest.mark.parametrize("T,d,E,bias", [(129, 256, 8, False), (300, 2048, 128, True), (64, 72, 5, True)])
def test_router_logits_and_backward(T, d, E, bias):
    w = wl.small_workload(T=T, d=d, E=E, k=1, h=64, routing="learned", zipf=bias)
    inp = wl.generate(w, seed=3)
    x = bf16_tensor(inp["x"], DEV)
    Wr = torch.from_numpy(inp["W_r"]).to(DEV)
    b = torch.from_numpy(inp["b"]).to(DEV) if bias else None
    z = torch.empty(T, E, dtype=torch.float32, device=DEV)
    L.moe_router_logits(x, Wr, b, z)
    zref = ol.router_logits(inp["x"], inp["W_r"], inp.get("b"), np.float64)
    assert_close(z, zref, "logits", rel_l2=1e-5, max_abs=1e-5)
    rng = np.random.default_rng(4)
    dz = rng.standard_normal((T, E)).astype(np.float32)
    dx0 = rng.standard_normal((T, d)).astype(np.float32)
    dx = bf16_tensor(wl.bf16_bits(dx0), DEV)
    dWr = torch.empty(d, E, dtype=torch.float32, device=DEV)
    db = torch.empty(E, dtype=torch.float32, device=DEV)
    L.moe_router_logits_bwd(x, Wr, torch.from_numpy(dz).to(DEV), dx, dWr, db, _ws(T, E, 1, d))
    dxr, dWref, dbref = ol.router_logits_backward(inp["x"], inp["W_r"], dz)
    assert_close(dx, ol.decode_bf16(wl.bf16_bits(dx0)) + dxr, "dx")
    assert_close(dWr, dWref, "dW_r", rel_l2=1e-5, max_abs=1e-5)
    assert_close(db, dbref, "db", rel_l2=1e-5, max_abs=1e-5)


@pytest.mark.parametrize("T,d,E,bias", [(129, 256, 8, False), (300, 2048, 128, True), (64, 72, 5, True),
                                        (1000, 512, 300, True), (16384, 2048, 128, True)])
def test_router_logits_tensor_cores(T, d, E, bias):
    # the tcgen05 router (W_r split into three bf16 parts, fp32 accumulation)
    # against the fp64 oracle at the fp32 router tolerance: ragged rows (129,
    # 300), a K tail (d = 72), expert tiles cut short (E = 5, 300), full size
    w = wl.small_workload(T=T, d=d, E=E, k=1, h=64, routing="learned", zipf=bias)
    inp = wl.generate(w, seed=7, with_backward=False)
    x = bf16_tensor(inp["x"], DEV)
    Wr = torch.from_numpy(inp["W_r"]).to(DEV)
    b = torch.from_numpy(inp["b"]).to(DEV) if bias else None
    z = torch.full((T, E), float("nan"), dtype=torch.float32, device=DEV)
    ws = _ws(T, E, 1, d)
    L.moe_reset_status(ws)
    L.moe_router_logits_tc(x, Wr, b, z, ws)
    assert L.moe_get_status(ws) == 0
    zref = ol.router_logits(inp["x"], inp["W_r"], inp.get("b"), np.float64)
    assert_close(z, zref, "logits", rel_l2=1e-5, max_abs=1e-5)


@pytest.mark.parametrize("T,d,E,k,bias", [(129, 256, 8, 2, False), (300, 2048, 128, 4, True),
                                          (64, 72, 5, 3, True), (3000, 128, 16, 8, False),
                                          (16384, 2048, 128, 4, True)])
def test_router_backward_through_topk(T, d, E, k, bias):
    # backward of the router GEMM when only the selected logits carry gradient:
    # against the fp64 oracle and against the dense call on the same d_logits;
    # the Zipf bias leaves experts empty, whose dW_r columns and db must be 0
    w = wl.small_workload(T=T, d=d, E=E, k=k, h=64, routing="learned", zipf=bias)
    inp = wl.generate(w, seed=8, with_backward=False)
    z = ol.router_logits(inp["x"], inp["W_r"], inp.get("b"))
    idx = ol.topk(z, k)
    g = ol.topk_gates(z, idx)
    rng = np.random.default_rng(9)
    dz = ol.router_topk_backward(g, rng.standard_normal((T, k)), idx, E).astype(np.float32)
    counts, _, _, _ = ol.route_map(idx, E)
    x = bf16_tensor(inp["x"], DEV)
    Wr = torch.from_numpy(inp["W_r"]).to(DEV)
    dzt = torch.from_numpy(dz).to(DEV)
    it = torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    cnt, off = torch.empty(E, **i32), torch.empty(E + 1, **i32)
    ros, sor = torch.empty(T * k, **i32), torch.empty(T * k, **i32)
    ws = _ws(T, E, k, d)
    L.moe_expert_offsets(it, E, cnt, off, ros, sor, ws)
    dx0 = wl.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    dx = bf16_tensor(dx0, DEV)
    dWr = torch.full((d, E), float("nan"), dtype=torch.float32, device=DEV)
    db = torch.full((E,), float("nan"), dtype=torch.float32, device=DEV)
    L.moe_router_logits_bwd_topk(x, Wr, dzt, it, off, sor, dx, dWr, db, ws)
    dxr, dWref, dbref = ol.router_logits_backward(inp["x"], inp["W_r"], dz)
    assert_close(dx, ol.decode_bf16(dx0) + dxr, "dx")
    assert_close(dWr, dWref, "dW_r", rel_l2=1e-5, max_abs=1e-5)
    assert_close(db, dbref, "db", rel_l2=1e-5, max_abs=1e-5)
    empty = np.flatnonzero(counts == 0)
    assert torch.count_nonzero(dWr[:, torch.from_numpy(empty).to(DEV)]).item() == 0
    assert torch.count_nonzero(db[torch.from_numpy(empty).to(DEV)]).item() == 0
    # the dense call on the same (zero-padded) d_logits
    dx2 = bf16_tensor(dx0, DEV)
    dWr2 = torch.empty(d, E, dtype=torch.float32, device=DEV)
    db2 = torch.empty(E, dtype=torch.float32, device=DEV)
    L.moe_router_logits_bwd(x, Wr, dzt, dx2, dWr2, db2, _ws(T, E, k, d))
    assert_close(dWr, dWr2.cpu().numpy(), "dW_r vs dense", rel_l2=1e-5, max_abs=1e-5)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (5, 2, 3), (1000, 4, 8), (4096, 4, 128),
                                   (3000, 8, 1024), (257, 2, 700), (16384, 4, 128),
                                   # many chunk histograms per expert group of the scan
                                   (65536, 4, 128), (40000, 8, 33), (33000, 8, 8)])
def test_route_map_bit_exact(T, k, E):
    rng = np.random.default_rng(T + E)
    if E >= 64:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    else:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if E > 4:
        idx[idx == 2] = 3        # expert 2 empty; some tokens now hit expert 3 twice
    dev = torch.from_numpy(idx).to(DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    ros = torch.empty(T * k, dtype=torch.int32, device=DEV)
    sor = torch.empty(T * k, dtype=torch.int32, device=DEV)
    ws = _ws(T, E, k)
    L.moe_expert_offsets(dev, E, counts, offs, ros, sor, ws)
    c, o, r, s = ol.route_map(idx, E)
    assert np.array_equal(i32(counts), c)
    assert np.array_equal(i32(offs), o)
    assert np.array_equal(i32(ros), r)
    assert np.array_equal(i32(sor), s)
    assert L.moe_get_status(ws) == 0


def test_route_map_empty_experts_and_zero_tokens():
    E, k = 16, 2
    idx = np.array([[0, 5], [5, 0], [15, 5]], np.int32)       # 13 empty experts
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    ros = torch.empty(6, dtype=torch.int32, device=DEV)
    sor = torch.empty(6, dtype=torch.int32, device=DEV)
    L.moe_expert_offsets(torch.from_numpy(idx).to(DEV), E, counts, offs, ros, sor, _ws(3, E, k))
    c, o, r, s = ol.route_map(idx, E)
    assert np.array_equal(i32(offs), o) and np.array_equal(i32(ros), r)
    # T = 0: counts and offsets are zero, nothing else touched
    counts.fill_(9); offs.fill_(9)
    L.moe_expert_offsets(torch.empty(0, k, dtype=torch.int32, device=DEV), E, counts, offs,
                         torch.empty(0, dtype=torch.int32, device=DEV),
                         torch.empty(0, dtype=torch.int32, device=DEV), _ws(0, E, k))
    assert np.all(i32(counts) == 0) and np.all(i32(offs) == 0)


def test_bad_expert_id_sets_device_status_without_faulting():
    E, k, T = 8, 2, 50
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[17, 1] = E + 3
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    ros = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    sor = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    ws = _ws(T, E, k)
    L.moe_reset_status(ws)
    L.moe_expert_offsets(torch.from_numpy(idx).to(DEV), E, counts, offs, ros, sor, ws)
    assert L.moe_get_status(ws) == 1            # MOE_DEV_BAD_EXPERT_ID
    assert i32(counts).sum() == T * k - 1
    torch.cuda.synchronize()                     # the context is still healthy
    L.moe_reset_status(ws)
    assert L.moe_get_status(ws) == 0
    # the bad slot takes no row; every valid slot keeps its oracle row
    bad = 17 * k + 1
    rows = i32(ros)
    assert rows[bad] == -1
    good = np.ones(T * k, bool); good[bad] = False
    # the valid slots in slot order form a route map of their own (k = 1)
    flat = idx.reshape(-1)
    _, _, expect, _ = ol.route_map(flat[good].reshape(-1, 1), E)
    assert np.array_equal(rows[good], expect)
    # the row kernels run on the map with the -1 entry and stay inside their
    # buffers (guard bands of sentinel rows on both sides)
    d, G = 64, 4
    rng = np.random.default_rng(6)
    x = bf16_tensor(wl.bf16_bits(rng.standard_normal((T, d)).astype(np.float32)), DEV)
    g = torch.from_numpy(rng.random((T, k)).astype(np.float32)).to(DEV)
    sent = torch.full(((T * k + 2 * G), d), 7.0, dtype=torch.bfloat16, device=DEV)
    xp = sent[G:G + T * k]
    L.moe_dispatch_rows(x, ros, k, xp)
    yp_full = torch.full(((T * k + 2 * G), d), 7.0, dtype=torch.bfloat16, device=DEV)
    yp = yp_full[G:G + T * k]
    yp.copy_(xp)
    out_full = torch.full((T + 2 * G, d), 7.0, dtype=torch.bfloat16, device=DEV)
    out = out_full[G:G + T]
    L.moe_combine(yp, ros, g, k, out)
    dyp_full = torch.full(((T * k + 2 * G), d), 7.0, dtype=torch.bfloat16, device=DEV)
    dyp = dyp_full[G:G + T * k]
    dg = torch.full((T, k), 5.0, dtype=torch.float32, device=DEV)
    L.moe_combine_bwd(x, yp, ros, g, k, dyp, dg)
    xq_full = torch.full(((T * k + 2 * G), d), 9, dtype=torch.uint8, device=DEV)
    xs_full = torch.full(((T * k + 2 * G), d // 32), 9, dtype=torch.uint8, device=DEV)
    L.moe_dispatch_rows_mxfp8(x, ros, k, xq_full[G:G + T * k], xs_full[G:G + T * k])
    torch.cuda.synchronize()
    for name, full, n in (("xp", sent, T * k), ("out", out_full, T), ("dyp", dyp_full, T * k)):
        f = as_f64(full)
        assert np.all(f[:G] == 7.0) and np.all(f[G + n:] == 7.0), name
    for name, full in (("xq", xq_full), ("xs", xs_full)):
        f = full.cpu().numpy()
        assert np.all(f[:G] == 9) and np.all(f[G + T * k:] == 9), name
    # valid slots: exact copies and sums of the oracle's; the bad slot adds 0
    xf = as_f64(x)
    assert np.array_equal(as_f64(xp)[rows[good]], np.repeat(xf, k, axis=0)[good])
    gg = as_f64(g).copy(); gg[17, 1] = 0.0
    ref_out = ol.combine(as_f64(yp), rows.clip(0), gg, k)
    assert_close(out, ref_out, "combine with a skipped slot")
    assert as_f64(dg)[17, 1] == 0.0
    assert L.moe_get_status(ws) == 0


# k = 3 and 6 take two 16-byte vectors a row a pass (k = 4 too); d = 264 and
# 520 leave a ragged last pass, d = 8 a single vector a row
@pytest.mark.parametrize("T,d,k", [(1, 8, 1), (333, 2048, 4), (1024, 264, 2), (97, 4096, 8),
                                   (129, 264, 3), (64, 8, 3), (50, 520, 6)])
def test_dispatch_exact_and_combine(T, d, k):
    E = 16
    rng = np.random.default_rng(T * 3 + d)
    x = wl.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    c, o, ros, sor = ol.route_map(idx, E)
    xt = bf16_tensor(x, DEV)
    rost = torch.from_numpy(ros).to(DEV)
    xp = torch.empty(T * k, d, dtype=torch.bfloat16, device=DEV)
    L.moe_dispatch_rows(xt, rost, k, xp)
    assert np.array_equal(as_f64(xp), ol.dispatch(x, ros, k))        # exact copy
    # identity experts and unit gates: combine returns k * x exactly
    out = torch.empty(T, d, dtype=torch.bfloat16, device=DEV)
    L.moe_combine(xp, rost, torch.ones(T, k, dtype=torch.float32, device=DEV), k, out)
    if k in (1, 2, 4, 8):
        assert np.array_equal(as_f64(out), k * ol.decode_bf16(x))
    # weighted combine and the unpermute-sum (gates = None)
    yp = wl.bf16_bits(rng.standard_normal((T * k, d)).astype(np.float32))
    g = rng.random((T, k)).astype(np.float32)
    ypt = bf16_tensor(yp, DEV)
    L.moe_combine(ypt, rost, torch.from_numpy(g).to(DEV), k, out)
    assert_close(out, ol.combine(yp, ros, g, k), "combine")
    L.moe_combine(ypt, rost, None, k, out)
    assert_close(out, ol.unpermute_sum(yp, ros, k), "unpermute")
    # combine backward
    dout = wl.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    dyp = torch.empty(T * k, d, dtype=torch.bfloat16, device=DEV)
    dg = torch.empty(T, k, dtype=torch.float32, device=DEV)
    L.moe_combine_bwd(bf16_tensor(dout, DEV), ypt, rost, torch.from_numpy(g).to(DEV), k, dyp, dg)
    dyp_ref, dg_ref = ol.combine_backward(dout, yp, ros, g, k)
    assert_close(dyp, dyp_ref, "dyp")
    assert_close(dg, dg_ref, "dgate", rel_l2=1e-5, max_abs=1e-5)
