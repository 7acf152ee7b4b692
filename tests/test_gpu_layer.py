"""GPU parity of the whole layer (forward + backward) against the fp64 oracle.

Small problems are compared tensor by tensor; the full-size workloads are
compared bit-exactly on the routing metadata and on sampled tokens and
experts that the oracle recomputes one by one.  Learned routers: both sides
route on the oracle's fp32 logits, passed to the device top-k through the C
ABI; the device's own logits GEMM is compared with tolerance."""
import numpy as np
import pytest
import torch

import oracle.layer as ol
from token_dispatch_grouped_router_gb300 import libmoe as L
from token_dispatch_grouped_router_gb300 import workloads as wl
from token_dispatch_grouped_router_gb300.layer import HostPipeline, MoELayer, bf16_tensor

from gpu_helpers import assert_close, as_f64, ensure_built, i32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    L.load()


def make_layer(w, inp, backward=True, logits=None):
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=(w.routing == "learned"),
                     device=DEV, with_backward=backward)
    layer.load_inputs(inp)
    if w.routing == "learned":
        layer.load_logits(logits if logits is not None
                          else ol.router_logits(inp["x"], inp["W_r"], inp.get("b")))
    return layer


def run(layer, backward=True):
    L.moe_reset_status(layer.ws)
    layer.forward()
    if backward:
        layer.backward()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0


def compare_full(layer, w, inp, backward=True):
    z = None
    if w.routing == "learned":
        z = layer.logits.cpu().numpy()
    ref = ol.layer_forward(inp, w.k, w.E, logits=z)
    assert np.array_equal(i32(layer.idx), ref["idx"])
    assert np.array_equal(i32(layer.counts), ref["counts"])
    assert np.array_equal(i32(layer.offsets), ref["offsets"])
    assert np.array_equal(i32(layer.row_of_slot), ref["row_of_slot"])
    assert np.array_equal(i32(layer.slot_of_row), ref["slot_of_row"])
    assert np.array_equal(as_f64(layer.xp), ref["Xp"])
    assert_close(layer.gate, ref["g"], "gate", rel_l2=1e-6, max_abs=1e-6)
    for n, key in (("h1", "H1"), ("h3", "H3"), ("a", "A"), ("yp", "Yp"), ("out", "out")):
        assert_close(getattr(layer, n), ref[key], n)
    if not backward:
        return ref, None
    refb = ol.layer_backward(inp, ref, w.k, w.E)
    for n, key in (("dyp", "dYp"), ("dgate", "dg"), ("dh1", "dH1"), ("dh3", "dH3"),
                   ("dxp", "dXp"), ("dW1", "dW1"), ("dW3", "dW3"), ("dW2", "dW2"),
                   ("dX", "dX"), ("dlogits", "dz")):
        assert_close(getattr(layer, n), refb[key], n)
    if w.routing == "learned":
        assert_close(layer.dW_r, refb["dW_r"], "dW_r")
        assert_close(layer.db, refb["db"], "db")
    # an expert with no rows gets exactly zero weight gradients
    for e in np.nonzero(ref["counts"] == 0)[0]:
        for n in ("dW1", "dW3", "dW2"):
            assert torch.count_nonzero(getattr(layer, n)[e]).item() == 0, (n, e)
    return ref, refb


@pytest.mark.parametrize("T,d,E,k,h,empty", [
    (300, 128, 6, 2, 192, (3,)),        # ragged rows, h not a multiple of 128
    (200, 256, 3, 1, 64, ()),           # one 64-wide hidden tile
    (513, 192, 8, 4, 320, (0, 7)),      # d and h off the 256 grid, empty ends
    (1000, 512, 16, 4, 256, (5,)),      # several tiles per expert
    (64, 128, 1, 1, 128, ()),           # a single dense expert
    # >= 512 rows per expert on average: the UP, DOWN and DX GEMMs run on
    # CTA pairs with 256-row tiles
    (2700, 192, 4, 2, 320, (2,)),       # pair tiles, ragged tails, one empty expert
    (2100, 256, 2, 1, 128, ()),         # pair tiles, one 128-wide hidden tile
    (1100, 128, 1, 1, 64, ()),          # last tile's odd CTA holds no rows
    (1000, 256, 8, 8, 192, ()),         # top-8 of 8: every token in every expert
    # the weight-gradient tiles split along the rows (fp32 partials, ordered
    # sum) with an empty expert among them
    (3000, 256, 3, 1, 256, (0,)),
    # more experts than DA's CTA-pair tile table holds: DA on single CTAs
    # beside the CTA-pair UP, DOWN, DX and wgrad GEMMs
    (31000, 64, 240, 4, 64, ()),
    # one expert holds every row: the weight gradient's plan has fewer work
    # units (3) than pairs, and the other experts' zero tiles go to the pairs
    # that stay (single-CTA, then CTA-pair row GEMMs)
    (600, 256, 8, 1, 256, (0, 1, 2, 4, 5, 6, 7)),
    (2100, 256, 4, 1, 256, (0, 1, 3)),
])
def test_layer_small_full_compare(T, d, E, k, h, empty):
    w = wl.small_workload(T=T, d=d, E=E, k=k, h=h)
    inp = wl.generate(w, seed=1)
    if empty:
        keep = [e for e in range(E) if e not in empty]
        rng = np.random.default_rng(2)
        inp["idx"] = np.stack([rng.permutation(keep)[:k] for _ in range(T)]).astype(np.int32)
    layer = make_layer(w, inp)
    run(layer)
    ref, _ = compare_full(layer, w, inp)
    for e in empty:
        assert ref["counts"][e] == 0


def test_layer_learned_router_zipf_full_compare():
    w = wl.small_workload(T=640, d=256, E=32, k=4, h=192, routing="learned", zipf=True)
    inp = wl.generate(w, seed=0)
    layer = make_layer(w, inp)
    run(layer)
    ref, _ = compare_full(layer, w, inp)
    assert (ref["counts"] == 0).sum() >= 1 and ref["counts"].max() > 4 * ref["counts"].mean()


def test_tiny_workload_forward_full_compare():
    w = wl.get_workload("tiny_e8")
    inp = wl.generate(w, seed=0)
    layer = make_layer(w, inp, backward=False)
    run(layer, backward=False)
    compare_full(layer, w, inp, backward=False)
    # the device's own router GEMM matches the oracle's logits
    zdev = torch.empty_like(layer.logits)
    L.moe_router_logits(layer.x, layer.W_r, layer.b, zdev)
    assert_close(zdev, ol.router_logits(inp["x"], inp["W_r"], None, np.float64), "logits",
                 rel_l2=1e-5, max_abs=1e-5)


def test_graph_capture_proves_no_host_sync_and_replays_bitwise():
    w = wl.small_workload(T=700, d=256, E=8, k=2, h=128, routing="learned", zipf=True)
    inp = wl.generate(w, seed=4)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=True, device=DEV)
    layer.load_inputs(inp)
    layer.step()                 # eager reference (device router logits included)
    torch.cuda.synchronize()
    eager = {n: getattr(layer, n).clone() for n in ("idx", "offsets", "out", "dX", "dW1", "dW2", "dW_r")}
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        # any host synchronisation or device->host copy inside would break capture
        with torch.cuda.graph(g, stream=s):
            layer.step()
    for buf in ("out", "dX", "dW1", "dW2", "dW_r"):
        getattr(layer, buf).zero_()
    g.replay()
    torch.cuda.synchronize()
    for n, v in eager.items():
        assert torch.equal(getattr(layer, n), v), n


@pytest.mark.parametrize("routing,factor", [("uniform", None), ("learned", None), ("learned", 1.25)])
def test_second_stream_backward_equals_one_stream_bitwise(routing, factor):
    # with side_stream=True the unpermute and the router backward run on a
    # second stream beside the weight-gradient GEMM (the padded layer's
    # unpadded route map after it); the results equal the single-stream step
    # bit for bit, also with three steps queued back to back (each step's
    # forward after the last join)
    w = wl.small_workload(T=2304, d=256, E=8, k=4, h=256, routing=routing,
                          zipf=(routing == "learned"))
    inp = wl.generate(w, seed=9)
    names = ("out", "dgate", "dlogits", "dxp", "dW1", "dW3", "dW2", "dX")
    if routing == "learned":
        names += ("dW_r", "db")
    res = []
    for side in (False, True):
        layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=(routing == "learned"), device=DEV,
                         capacity_factor=factor, side_stream=side)
        assert (layer._side is not None) == side
        layer.load_inputs(inp)
        L.moe_reset_status(layer.ws)
        for _ in range(3):
            layer.step()
        torch.cuda.synchronize()
        assert L.moe_get_status(layer.ws) == 0
        res.append({n: getattr(layer, n).clone() for n in names})
    for n in names:
        assert torch.equal(res[0][n], res[1][n]), n
    # the fork and the join capture into a CUDA graph and replay bit for bit
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            layer.step()
    for n in names:
        getattr(layer, n).zero_()
    g.replay()
    torch.cuda.synchronize()
    for n in names:
        assert torch.equal(getattr(layer, n), res[1][n]), n


@pytest.mark.parametrize("T,E", [(2000, 16), (2048, 4)])   # single-CTA / CTA-pair row GEMMs
def test_deterministic_bitwise(T, E):
    w = wl.small_workload(T=T, d=256, E=E, k=4, h=256)
    inp = wl.generate(w, seed=5)
    layer = make_layer(w, inp)
    run(layer)
    first = {n: getattr(layer, n).clone() for n in ("out", "dgate", "dxp", "dW1", "dW3", "dW2", "dX")}
    run(layer)
    for n, v in first.items():
        assert torch.equal(getattr(layer, n), v), n


@pytest.mark.parametrize("T,E", [(2000, 16), (2048, 4)])   # single-CTA / CTA-pair row GEMMs
def test_recompute_backward_matches_saved_bitwise(T, E):
    # the recompute policy gathers Xp again and recomputes H1, H3, A in the
    # backward; with those buffers poisoned after the forward it must still
    # reproduce the saved-activation step bit for bit
    w = wl.small_workload(T=T, d=256, E=E, k=4, h=256)
    inp = wl.generate(w, seed=7)
    layer = make_layer(w, inp)
    run(layer)
    names = ("out", "dgate", "dh1", "dh3", "dxp", "dW1", "dW3", "dW2", "dX")
    saved = {n: getattr(layer, n).clone() for n in names}
    layer.recompute = True
    L.moe_reset_status(layer.ws)
    layer.forward()
    for n in ("xp", "h1", "h3", "a"):
        getattr(layer, n).fill_(float("nan"))
    layer.backward()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    for n, v in saved.items():
        assert torch.equal(getattr(layer, n), v), n
    # and the recomputed step against the fp64 oracle, tensor by tensor (the
    # recomputed Xp, H1, H3, A included)
    compare_full(layer, w, inp)


@pytest.mark.parametrize("T,E", [(333, 5), (1400, 2)])    # single-CTA / CTA-pair row GEMMs
def test_outputs_stay_inside_their_buffers(T, E):
    # every output is a view at the front of a larger buffer whose tail holds a
    # sentinel; a write past the end of any output would change it
    w = wl.small_workload(T=T, d=192, E=E, k=2, h=320)
    inp = wl.generate(w, seed=6)
    layer = make_layer(w, inp)
    guards = {}
    for n in ("xp", "h1", "h3", "a", "yp", "out", "dyp", "dgate", "dh1", "dh3", "dxp", "dW1",
              "dW3", "dW2", "dX", "dlogits", "row_of_slot", "slot_of_row", "counts", "offsets"):
        t = getattr(layer, n)
        big = torch.empty(t.numel() + 4096, dtype=t.dtype, device=DEV)
        big.view(torch.uint8)[:].fill_(0xA5)
        view = big[:t.numel()].view(t.shape)
        view.copy_(t)
        setattr(layer, n, view)
        guards[n] = big
    run(layer)
    for n, big in guards.items():
        tail = big[-4096:].view(torch.uint8)
        assert bool((tail == 0xA5).all()), f"{n} written past its end"
    compare_full(layer, w, inp)


def test_zero_tokens_gives_zero_weight_gradients():
    w = wl.small_workload(T=0, d=128, E=4, k=2, h=128)
    layer = MoELayer(0, 128, 4, 2, 128, learned=False, device=DEV)
    for n in ("W1", "W3", "W2"):
        getattr(layer, n).normal_()
    for n in ("dW1", "dW3", "dW2"):
        getattr(layer, n).fill_(1.0)
    run(layer)
    for n in ("dW1", "dW3", "dW2"):
        assert torch.count_nonzero(getattr(layer, n)).item() == 0
    assert i32(layer.offsets).sum() == 0


def test_argument_errors_on_device_buffers():
    x = torch.zeros(8, 96, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(2, 96, 128, dtype=torch.bfloat16, device=DEV)
    W2 = torch.zeros(2, 128, 96, dtype=torch.bfloat16, device=DEV)
    o = torch.zeros(3, dtype=torch.int32, device=DEV)
    hbuf = torch.zeros(8, 128, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(L.MoEError) as ei:
        L.moe_grouped_swiglu_fwd(x, o, W, W, W2, hbuf, hbuf, hbuf, x, ws)
    assert ei.value.status == -2           # d = 96 is not a multiple of 64
    torch.cuda.synchronize()


# ------------------------------------------------------- full-size workloads

def _sampled_reference(inp, w, idx, g, ros, toks, hs, experts):
    """Oracle values for the sampled tokens (forward + backward rows) and for
    sampled hidden units of the sampled experts' weight gradients."""
    k = w.k
    x = ol.decode_bf16(inp["x"]); dY = ol.decode_bf16(inp["dY"])
    res = {"yp": [], "h1": [], "out": [], "dxp": [], "dgate": [], "dX": [], "rows": []}
    for t in toks:
        rows = ros[t * k:(t + 1) * k]
        out_t = np.zeros(w.d); dX_t = np.zeros(w.d)
        dg_t = np.zeros(k)
        for j in range(k):
            e = int(idx[t, j])
            f = ol.expert_ffn_forward(x[t:t + 1], [0, 1], inp["W1"][e:e + 1],
                                      inp["W3"][e:e + 1], inp["W2"][e:e + 1])
            dyp = g[t, j] * dY[t:t + 1]
            b = ol.expert_ffn_backward(x[t:t + 1], [0, 1], inp["W1"][e:e + 1],
                                       inp["W3"][e:e + 1], inp["W2"][e:e + 1],
                                       f["H1"], f["H3"], f["A"], dyp)
            res["yp"].append(f["Yp"][0]); res["h1"].append(f["H1"][0]); res["dxp"].append(b["dXp"][0])
            res["rows"].append(int(rows[j]))
            out_t += g[t, j] * f["Yp"][0]
            dX_t += b["dXp"][0]
            dg_t[j] = float(dY[t] @ f["Yp"][0])
        if "W_r" in inp:
            # learned router: dX also carries dz W_r^T through the top-k softmax
            dz = ol.router_topk_backward(g[t:t + 1], dg_t[None], idx[t:t + 1], w.E)
            dX_t += ol.router_logits_backward(x[t:t + 1], inp["W_r"], dz)[0][0]
        res["out"].append(out_t); res["dX"].append(dX_t); res["dgate"].append(dg_t)
    # weight gradients of sampled experts, restricted to hidden units hs
    wg = {}
    c, off, _, sor = ol.route_map(idx, w.E)
    for e in experts:
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            wg[e] = None
            continue
        slots = sor[lo:hi].astype(np.int64)
        X = x[slots // k]
        dyp = g[slots // k, slots % k][:, None] * dY[slots // k]
        W1s = inp["W1"][e][:, hs][None]; W3s = inp["W3"][e][:, hs][None]
        W2s = inp["W2"][e][hs, :][None]
        f = ol.expert_ffn_forward(X, [0, hi - lo], W1s, W3s, W2s)
        b = ol.expert_ffn_backward(X, [0, hi - lo], W1s, W3s, W2s, f["H1"], f["H3"], f["A"], dyp)
        wg[e] = (b["dW1"][0], b["dW3"][0], b["dW2"][0])
    return res, wg


@pytest.mark.parametrize("key", ["dense_e8", "pool_e128", "skew_e128", "train_e128",
                                 "max_experts_top8"])
def test_full_size_sampled(key):
    if key == "max_experts_top8":
        # the largest expert count the library takes, top-8 routing, 512 rows per
        # expert: pair GEMMs and a K-split wgrad with 1024-expert tile tables
        w = wl.small_workload(T=65536, d=128, E=1024, k=8, h=128)
    else:
        w = wl.get_workload(key)
    inp = wl.generate(w, seed=0)
    zref = None
    if w.routing == "learned":
        zref = ol.router_logits(inp["x"], inp["W_r"], inp.get("b"))
    layer = make_layer(w, inp, logits=zref)
    run(layer)
    # routing metadata, bit-exact over the whole step
    if w.routing == "learned":
        idx = ol.topk(zref, w.k)
        g = ol.topk_gates(zref, idx)
    else:
        idx = inp["idx"]
        g = ol.softmax_gates(inp["glogit"])
    c, off, ros, sor = ol.route_map(idx, w.E)
    assert np.array_equal(i32(layer.idx), idx)
    assert np.array_equal(i32(layer.counts), c) and np.array_equal(i32(layer.offsets), off)
    assert np.array_equal(i32(layer.row_of_slot), ros) and np.array_equal(i32(layer.slot_of_row), sor)
    assert_close(layer.gate, g, "gate", rel_l2=1e-6, max_abs=1e-6)
    rng = np.random.default_rng(7)
    toks = np.sort(rng.choice(w.T, 24, replace=False))
    hs = np.sort(rng.choice(w.h, 16, replace=False))
    nonempty = np.nonzero(c)[0]
    experts = sorted({int(nonempty[np.argmax(c[nonempty])]), int(nonempty[np.argmin(c[nonempty])]),
                      int(rng.choice(nonempty))} | set(int(e) for e in np.nonzero(c == 0)[0][:1]))
    res, wg = _sampled_reference(inp, w, idx, g, ros, toks, hs, experts)
    rows = torch.tensor(res["rows"], device=DEV, dtype=torch.long)
    tk = torch.tensor(toks, device=DEV, dtype=torch.long)
    # dispatch is an exact copy
    xp_rows = as_f64(layer.xp[rows])
    assert np.array_equal(xp_rows, ol.decode_bf16(inp["x"])[np.repeat(toks, w.k)])
    assert_close(layer.yp[rows], np.array(res["yp"]), "yp")
    assert_close(layer.h1[rows], np.array(res["h1"]), "h1")
    assert_close(layer.out[tk], np.array(res["out"]), "out")
    assert_close(layer.dxp[rows], np.array(res["dxp"]), "dxp")
    assert_close(layer.dgate[tk], np.array(res["dgate"]), "dgate")
    assert_close(layer.dX[tk], np.array(res["dX"]), "dX")
    hst = torch.tensor(hs, device=DEV, dtype=torch.long)
    for e, v in wg.items():
        if v is None:
            for n in ("dW1", "dW3", "dW2"):
                assert torch.count_nonzero(getattr(layer, n)[e]).item() == 0
            continue
        assert_close(layer.dW1[e][:, hst], v[0], f"dW1[{e}]")
        assert_close(layer.dW3[e][:, hst], v[1], f"dW3[{e}]")
        assert_close(layer.dW2[e][hst, :], v[2], f"dW2[{e}]")
    if w.routing == "learned":
        # the device's own router GEMM agrees with the oracle's logits
        zdev = torch.empty_like(layer.logits)
        L.moe_router_logits(layer.x, layer.W_r, layer.b, zdev)
        zd = zdev[tk].cpu().numpy()
        assert_close(zd, ol.router_logits(ol.decode_bf16(inp["x"])[toks], inp["W_r"], inp["b"],
                                          np.float64), "logits", rel_l2=1e-5, max_abs=1e-5)


def test_combined_calls_equal_the_phase_calls():
    w = wl.small_workload(T=900, d=256, E=12, k=4, h=192)
    inp = wl.generate(w, seed=8)
    layer = make_layer(w, inp)
    run(layer)                     # phase by phase (fwd_up, fwd_down, bwd_dact, bwd_dx, bwd_wgrad)
    keep = {n: getattr(layer, n).clone() for n in ("h1", "h3", "a", "yp", "dh1", "dh3", "dxp",
                                                   "dW1", "dW3", "dW2")}
    for n in keep:
        getattr(layer, n).zero_()
    L.moe_grouped_swiglu_fwd(layer.xp, layer.offsets, layer.W1, layer.W3, layer.W2, layer.h1,
                             layer.h3, layer.a, layer.yp, layer.ws)
    L.moe_grouped_swiglu_bwd(layer.xp, layer.offsets, layer.W1, layer.W3, layer.W2, layer.h1,
                             layer.h3, layer.a, layer.dyp, layer.dh1, layer.dh3, layer.dxp,
                             layer.dW1, layer.dW3, layer.dW2, layer.ws)
    torch.cuda.synchronize()
    for n, v in keep.items():
        assert torch.equal(getattr(layer, n), v), n


def test_host_pipeline_matches_sequential_steps():
    # three steps with different token inputs: the pipelined runner, whose
    # input and output copies of neighbouring steps overlap the compute on
    # their own streams, must reproduce each step's results bit for bit
    w = wl.small_workload(T=1500, d=256, E=4, k=2, h=256)
    base = wl.generate(w, seed=11)
    steps = [base]
    for seed in (12, 13):
        other = wl.generate(w, seed=seed)
        steps.append({**base, **{n: other[n] for n in ("x", "dY", "idx", "glogit")}})
    layer = make_layer(w, base)
    ref = []
    for inp in steps:
        layer.load_inputs(inp)
        run(layer)
        ref.append({n: getattr(layer, n).cpu() for n in ("out", "dX")})
    hin = [{"x": bf16_tensor(i["x"], "cpu").pin_memory(),
            "dY": bf16_tensor(i["dY"], "cpu").pin_memory(),
            "idx": torch.from_numpy(i["idx"]).pin_memory(),
            "glogit": torch.from_numpy(i["glogit"]).pin_memory()} for i in steps]
    hout = [{n: torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory() for n in ("out", "dX")}
            for _ in steps]
    pipe = HostPipeline(layer, input_names=tuple(hin[0]), output_names=("out", "dX"))
    L.moe_reset_status(layer.ws)
    pipe.run(hin, hout)
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    for i, (r, o) in enumerate(zip(ref, hout)):
        for n in ("out", "dX"):
            assert torch.equal(r[n], o[n]), (i, n)
