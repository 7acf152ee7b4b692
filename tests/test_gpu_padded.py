"""GPU parity of the capacity-padded layer against the fp64 oracle's padded
reference (oracle/padded.py).

The padded layer is the alternative the device route map replaces: every
expert gets C rows, its first C routed slots in token order and then zero
rows, later slots are dropped, and the same grouped GEMMs run on all E * C
rows.  Integer outputs (the padded route map, the kept mask) are compared
bit-exactly; floating point at the bf16 tolerance of the other GPU tests."""
import numpy as np
import pytest
import torch

import oracle.layer as ol
import oracle.padded as pd
from token_dispatch_grouped_router_gb300 import libmoe as L
from token_dispatch_grouped_router_gb300 import workloads as wl
from token_dispatch_grouped_router_gb300.layer import MoELayer

from gpu_helpers import assert_close, as_f64, ensure_built, i32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    L.load()


def _layer(w, inp, factor, z=None):
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=(w.routing == "learned"), device=DEV,
                     capacity_factor=factor)
    layer.load_inputs(inp)
    if z is not None:
        layer.load_logits(z)
    L.moe_reset_status(layer.ws)
    layer.step()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    return layer


def _routing(w, inp, z):
    if w.routing == "learned":
        idx = ol.topk(z, w.k)
        return idx, ol.topk_gates(z, idx)
    return inp["idx"], ol.softmax_gates(inp["glogit"])


def _check_map(layer, idx, E, C):
    c, o, ros, sor, routed = pd.capacity_route_map(idx, E, C)
    assert np.array_equal(i32(layer.counts), c) and np.array_equal(i32(layer.offsets), o)
    assert np.array_equal(i32(layer.row_of_slot), ros)
    assert np.array_equal(i32(layer.slot_of_row), sor)
    assert np.array_equal(i32(layer.routed), routed)
    return c, ros


def _skewed_idx(T, E, k, seed):
    rng = np.random.default_rng(seed)
    p = np.linspace(3.0, 1.0, E); p /= p.sum()
    return np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,d,E,k,h,factor,routing", [
    (600, 128, 6, 2, 192, 1.0, "uniform"),     # single-CTA row GEMMs, drops at the hot experts
    (2700, 192, 4, 2, 320, 1.1, "uniform"),    # CTA-pair row GEMMs, ragged zero tails
    (640, 256, 32, 4, 192, 1.25, "learned"),   # Zipf router: empty experts, heavy drops
    (900, 256, 12, 4, 192, 4.0, "uniform"),    # capacity above every load: nothing dropped
])
def test_padded_layer_full_compare(T, d, E, k, h, factor, routing):
    w = wl.small_workload(T=T, d=d, E=E, k=k, h=h, routing=routing, zipf=(routing == "learned"))
    inp = wl.generate(w, seed=3)
    z = None
    if routing == "learned":
        z = ol.router_logits(inp["x"], inp["W_r"], inp.get("b"))
    else:
        inp["idx"] = _skewed_idx(T, E, k, seed=4)
    layer = _layer(w, inp, factor, z)
    C = layer.C
    assert C == pd.capacity(T, k, E, factor) and layer.R == E * C
    idx, g = _routing(w, inp, z)
    assert np.array_equal(i32(layer.idx), idx)
    c, ros = _check_map(layer, idx, E, C)
    x = ol.decode_bf16(inp["x"])
    # padded rows: exact copies of the kept tokens, zeros elsewhere
    xp = as_f64(layer.xp)
    kept = np.nonzero(ros >= 0)[0]
    assert np.array_equal(xp[ros[kept]], x[kept // k])
    zero_rows = np.setdiff1d(np.arange(E * C), ros[kept])
    assert np.all(xp[zero_rows] == 0) and np.all(as_f64(layer.dyp)[zero_rows] == 0)
    fwd = pd.padded_forward(inp["x"], idx, g, inp["W1"], inp["W3"], inp["W2"], E, C)
    assert np.array_equal(ros.reshape(-1, k) >= 0, fwd["kept"])
    if factor >= 4.0:
        assert fwd["dropped"] == 0
    else:
        assert fwd["dropped"] > 0
    assert_close(layer.out, fwd["out"], "out")
    bwd = pd.padded_backward(inp["x"], idx, g, inp["W1"], inp["W3"], inp["W2"], inp["dY"], E, C,
                             W_r=inp.get("W_r") if routing == "learned" else None)
    assert_close(layer.dgate, bwd["dg"], "dgate")
    assert np.all(as_f64(layer.dgate)[~fwd["kept"]] == 0)
    for n in ("dW1", "dW3", "dW2", "dX"):
        assert_close(getattr(layer, n), bwd[n], n)
    assert_close(layer.dlogits, bwd["dz"], "dlogits")
    if routing == "learned":
        assert_close(layer.dW_r, bwd["dW_r"], "dW_r")
        assert_close(layer.db, bwd["db"], "db")
    for e in np.nonzero(c == 0)[0]:              # an expert with only zero rows
        for n in ("dW1", "dW3", "dW2"):
            assert torch.count_nonzero(getattr(layer, n)[e]).item() == 0, (n, e)


@pytest.mark.parametrize("key", ["pool_e128", "skew_e128"])
def test_padded_full_size_sampled(key):
    # capacity 1.25 (640 rows per expert at T = 16384, k = 4, E = 128): the
    # padded map bit-exact over the whole step, sampled tokens against the oracle
    w = wl.get_workload(key)
    inp = wl.generate(w, seed=0)
    z = ol.router_logits(inp["x"], inp["W_r"], inp.get("b")) if w.routing == "learned" else None
    layer = _layer(w, inp, 1.25, z)
    C = layer.C
    assert C == 640
    idx, g = _routing(w, inp, z)
    c, ros = _check_map(layer, idx, w.E, C)
    kept = (ros >= 0).reshape(-1, w.k)
    rng = np.random.default_rng(8)
    dropped_tokens = np.nonzero(~kept.all(axis=1))[0]
    toks = np.sort(rng.choice(w.T, 20, replace=False))
    if dropped_tokens.size:
        toks = np.union1d(toks, rng.choice(dropped_tokens, 4, replace=False))
    x = ol.decode_bf16(inp["x"]); dY = ol.decode_bf16(inp["dY"])
    out_ref, dX_ref, dg_ref = [], [], []
    for t in toks:
        out_t = np.zeros(w.d); dX_t = np.zeros(w.d); dg_t = np.zeros(w.k)
        for j in range(w.k):
            if not kept[t, j]:
                continue
            e = int(idx[t, j])
            f = ol.expert_ffn_forward(x[t:t + 1], [0, 1], inp["W1"][e:e + 1], inp["W3"][e:e + 1],
                                      inp["W2"][e:e + 1])
            b = ol.expert_ffn_backward(x[t:t + 1], [0, 1], inp["W1"][e:e + 1], inp["W3"][e:e + 1],
                                       inp["W2"][e:e + 1], f["H1"], f["H3"], f["A"],
                                       g[t, j] * dY[t:t + 1])
            out_t += g[t, j] * f["Yp"][0]
            dX_t += b["dXp"][0]
            dg_t[j] = float(dY[t] @ f["Yp"][0])
        if w.routing == "learned":
            dz = ol.router_topk_backward(g[t:t + 1], dg_t[None], idx[t:t + 1], w.E)
            dX_t += ol.router_logits_backward(x[t:t + 1], inp["W_r"], dz)[0][0]
        out_ref.append(out_t); dX_ref.append(dX_t); dg_ref.append(dg_t)
    tk = torch.tensor(toks, device=DEV, dtype=torch.long)
    assert_close(layer.out[tk], np.array(out_ref), "out")
    assert_close(layer.dgate[tk], np.array(dg_ref), "dgate")
    assert_close(layer.dX[tk], np.array(dX_ref), "dX")


def test_padded_layer_zero_tokens_and_graph_capture():
    # T = 0: every expert holds one zero row; the weight gradients are zero
    layer = MoELayer(0, 128, 4, 2, 128, learned=False, device=DEV, capacity_factor=1.25)
    for n in ("W1", "W3", "W2"):
        getattr(layer, n).normal_()
    for n in ("dW1", "dW3", "dW2"):
        getattr(layer, n).fill_(1.0)
    L.moe_reset_status(layer.ws)
    layer.step()
    torch.cuda.synchronize()
    assert L.moe_get_status(layer.ws) == 0
    assert layer.C == 1 and np.all(i32(layer.counts) == 0)
    for n in ("dW1", "dW3", "dW2"):
        assert torch.count_nonzero(getattr(layer, n)).item() == 0
    # the padded step has no host synchronisation: it captures into a CUDA
    # graph and replays bit for bit (learned Zipf router, dropped slots)
    w = wl.small_workload(T=640, d=256, E=32, k=4, h=192, routing="learned", zipf=True)
    inp = wl.generate(w, seed=5)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=True, device=DEV, capacity_factor=1.25)
    layer.load_inputs(inp)
    layer.step()
    torch.cuda.synchronize()
    names = ("row_of_slot", "out", "dX", "dW1", "dW2", "dW_r", "dgate")
    eager = {n: getattr(layer, n).clone() for n in names}
    assert (i32(layer.row_of_slot) < 0).any()            # some slots dropped
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer.step()
    for n in ("out", "dX", "dW1", "dW2", "dW_r"):
        getattr(layer, n).zero_()
    g.replay()
    torch.cuda.synchronize()
    for n, v in eager.items():
        assert torch.equal(getattr(layer, n), v), n
