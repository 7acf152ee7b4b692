#!/usr/bin/env python3
"""Throughput of the single-GPU MoE expert layer, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload KEY] [--impl ours|reference]

One step = one pass of the whole layer over one batch: router gates (or
router GEMM + top-k), device route map, rowwise dispatch, grouped SwiGLU GEMMs
(up, down), combine, combine backward, grouped GEMM backward (dact, dx,
wgrad), unpermute-sum and router backward.  Inputs are seeded synthetic
tensors resident in HBM.  Between timed steps a 256 MB buffer is written to
flush the 129 MB L2 (twice over); every library call of a step is bracketed by CUDA events
on the launching stream, so the per-kernel times below come from the timed
steps themselves.  The unpermute and the router backward run on a second
stream beside the weight-gradient GEMM; their times come from that stream's
events, and the step ends after the streams have joined.

Rank 0 prints one JSON line.  Under torchrun (N > 1) every rank runs its own
token batch with its own copy of the experts (replicas, no collective in the
data path); the step time is the maximum over ranks and `value` counts the
tokens of all ranks.

`--impl reference` times the fp64 CPU oracle instead (rank 0 only), on token
samples of the same workload, and reports the same metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tok/s fwd+bwd at E=8..128, k=4; grouped-GEMM % peak; dispatch GB/s"
UNIT = "tok/s"
FLUSH_BYTES = 256 << 20   # twice the L2
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SOURCES = {
    "gemm": ["grouped_swiglu.cu", "gemm_common.cuh", "sm103_ptx.cuh", "common.cuh"],
    "rows": ["permute.cu", "common.cuh"],
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dense_e8")
    ap.add_argument("--compare", default="pool_e128",
                    help="second workload timed the same way (expert-count flatness); '' to skip")
    ap.add_argument("--skew-workload", default="skew_e128",
                    help="learned Zipf-biased router workload timed the same way (uneven experts); "
                         "'' to skip")
    ap.add_argument("--mxfp8-workload", default="train_e128",
                    help="workload of the BF16 vs MXFP8-forward comparison; '' to skip")
    ap.add_argument("--capacity-factor", type=float, default=1.25,
                    help="capacity factor of the padded layer timed beside each workload "
                         "(C = ceil(f*T*k/E)); 0 to skip")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="total CPU time budget of the --impl reference run")
    return ap.parse_args()


# --------------------------------------------------------------------- utils

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def allmax(v: float, device=None) -> float:
    """Maximum of v over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens per second: every rank processes its own batch, the
    step takes the slowest rank's time."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def sources_sha(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "token_dispatch_grouped_router_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def work_per_launch(w):
    """Algorithmic FLOPs (GEMMs) or bytes (row kernels) of one launch per label."""
    R, d, h, T, k = w.R, w.d, w.h, w.T, w.k
    flops = {"gemm_up": 2.0 * R * d * 2 * h, "gemm_down": 2.0 * R * h * d,
             "gemm_dact": 2.0 * R * d * h, "gemm_dx": 2.0 * R * 2 * h * d,
             "gemm_wgrad": 3 * 2.0 * R * d * h}
    bytes_ = {"dispatch": 2.0 * (T * d + R * d) + 4.0 * R,
              "combine": 2.0 * (R * d + T * d) + 8.0 * R,
              "combine_bwd": 2.0 * (T * d + 2 * R * d) + 12.0 * R,
              "unpermute": 2.0 * (R * d + T * d) + 4.0 * R}
    return flops, bytes_


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 50 ms), each stamped with the
    host time it was read, so the samples of the timed region can be picked."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_uuid):
        self.uuid = device_uuid
        self.rows = []
        self.proc = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)

    def window(self, t0, t1):
        """Summary of the samples read during [t0, t1] (a sample is read up to
        one interval after it was taken); the nearest later sample otherwise."""
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [r for t, r in self.rows if t0 <= t <= t1 + 0.05]
        how = "inside the timed region"
        if not inside:
            after = [r for t, r in self.rows if t > t1]
            inside = after[:1]
            how = "first sample after the timed region (region shorter than the interval)"
        if not inside:
            return None
        sm = [num(r[0]) for r in inside if num(r[0]) is not None]
        reasons = sorted({self.NAMES[i] for r in inside for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(inside[0][1]),
                "power_w_max": max((num(r[2]) or 0.0) for r in inside), "reasons": reasons,
                "samples": len(inside), "which": how, "interval_ms": 50}


def step_timings(events):
    """Per-step and per-call times from the marks of the timed steps.

    `events` holds, per step, the (label, event, stream) marks in the order the
    step made them; each mark was recorded on the stream that was current.
    A step lasts from the first to the last mark of the stream its first mark
    is on (the step's stream: its last mark follows the join of any second
    stream); a call lasts from its mark to the next mark on the same stream.
    Returns (step times, {label: [times]}, labels marked on another stream).
    """
    step_ms, per_label, side_labels = [], {}, set()
    for lst in events:
        main = lst[0][2]
        by_stream = {}
        for lab, ev, st in lst:
            by_stream.setdefault(st, []).append((lab, ev))
        side_labels |= {lab for lab, _, st in lst if st != main}
        seq = by_stream[main]
        step_ms.append(seq[0][1].elapsed_time(seq[-1][1]))
        for seq in by_stream.values():
            for (lab, ev), (_, nxt) in zip(seq[:-1], seq[1:]):
                per_label.setdefault(lab, []).append(ev.elapsed_time(nxt))
    return step_ms, per_label, side_labels


def capacity_stats(counts, T: int, k: int, E: int, factor: float = 1.25):
    """What a layer padded to one capacity per expert would do with these
    per-expert row counts: capacity ceil(factor*T*k/E), every expert keeping
    at most that many rows.  Host arithmetic on the device's counts."""
    import math
    C = int(math.ceil(factor * T * k / E))
    R = T * k
    dropped = int(sum(max(0, int(c) - C) for c in counts))
    return {"capacity_factor": factor, "capacity": C, "dropped_rows": dropped,
            "dropped_fraction": dropped / R, "padded_over_routed_rows": E * C / R}


# ----------------------------------------------------------------- our arm

def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if dist:
        dist.barrier()
    from token_dispatch_grouped_router_gb300 import libmoe as L
    from token_dispatch_grouped_router_gb300 import workloads as wl
    from token_dispatch_grouped_router_gb300.layer import HostPipeline, MoELayer, bf16_tensor
    L.load()

    peaks = measured_peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if dist:
            dist.barrier()

    def make_layer(w, inp, mxfp8=False, capacity_factor=None):
        layer = MoELayer(w.T, w.d, w.E, w.k, w.h, learned=(w.routing == "learned"), device=dev,
                         capacity_factor=capacity_factor)
        layer.load_inputs(inp)
        if mxfp8:
            layer.enable_mxfp8()
            layer.quantize_weights()
        return layer

    def timed_layer(layer, K, W, step=None, sample_clocks=False):
        """W warm-up steps, then K timed steps with an L2 flush between them
        and a CUDA event before every library call of every timed step."""
        step = step or layer.step
        sampler = ClockSampler(device_uuid(dev)) if (rank == 0 and sample_clocks) else None
        if sampler:
            sampler.start()                  # running before the warm-up steps
        for _ in range(W):
            step()
        torch.cuda.synchronize()
        L.moe_reset_status(layer.ws)
        # ---------------------------------------------------------- timed region
        events = []                          # per step: [(label, event, stream), ...]

        def new_mark(lst):
            def mark(label):
                # on the current stream: the layer runs part of its backward
                # on a second stream, whose calls are timed by its own events
                st = torch.cuda.current_stream()
                ev = torch.cuda.Event(enable_timing=True)
                ev.record(st)
                lst.append((label, ev, st.cuda_stream))
            return mark

        barrier()
        torch.cuda.synchronize()
        n0 = L.moe_launch_count()
        t_wall = time.perf_counter()
        for _ in range(K):
            flush.zero_()                    # L2 flush, outside the step's events
            lst = []
            step(new_mark(lst))
            events.append(lst)
        torch.cuda.synchronize()
        barrier()
        t_end = time.perf_counter()
        wall = t_end - t_wall
        launches = L.moe_launch_count() - n0
        clocks = None
        if sampler:
            time.sleep(0.15)
            sampler.stop()
            clocks = sampler.window(t_wall, t_end)
        status = L.moe_get_status(layer.ws)
        if status != 0:
            raise RuntimeError(f"device status {status} after the timed steps")
        step_ms, per_label, side_labels = step_timings(events)
        return {"ms_per_step": allmax(statistics.mean(step_ms), dev),
                "kernels_ms": {k: statistics.mean(v) for k, v in per_label.items()},
                "side_labels": sorted(side_labels),
                "launches": launches, "clocks": clocks, "wall_s": wall}

    def time_alone(fn, reps=5):
        """Mean event-timed duration of one library call run by itself, L2
        flushed before each (the calls the step runs beside another kernel
        get their roofline from this)."""
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.mean(ts)

    def tile_overhead(layer):
        """Rows the row-grouped GEMMs multiply beyond the T*k routed rows: each
        expert's last tile of 256 (CTA pairs) or 128 rows (single CTAs) is only
        partly filled.  Read from the device counts after the timed steps,
        with what a capacity-padded layer would drop from the same counts."""
        c = layer.counts.cpu().numpy().astype(np.int64)
        out = {f"tiles_{t}": float((-(-c // t) * t).sum() / layer.R - 1.0) for t in (256, 128)}
        out["capacity_padding"] = capacity_stats(c, layer.T, layer.k, layer.E)
        return out

    def timed(w, inp, K, W, with_e2e, sample_clocks=True):
        layer = make_layer(w, inp)
        res = timed_layer(layer, K, W, sample_clocks=sample_clocks)
        res["row_tile_overhead"] = tile_overhead(layer)
        if "unpermute" in res["side_labels"]:
            res["alone_ms"] = {"unpermute": time_alone(
                lambda: L.moe_combine(layer.dxp, layer.row_of_slot, None, layer.k, layer.dX))}
        if with_e2e:
            res["e2e"] = e2e(layer, inp, K)
            # the recompute policy (Xp gathered again, H1/H3/A recomputed in
            # the backward): time against activation memory
            layer.recompute = True
            res["recompute"] = timed_layer(layer, K, W)
            res["recompute"]["activation_bytes"] = layer.activation_bytes()
            layer.recompute = False
        del layer
        torch.cuda.empty_cache()
        if args.capacity_factor > 0:
            res["padded"] = timed_padded(w, inp, K, W, res["ms_per_step"])
        return res

    def timed_padded(w, inp, K, W, unpadded_ms):
        """The capacity-padded layer on the same inputs, timed the same way:
        every expert multiplies C rows (first C routed in token order, then
        zero rows), later slots are dropped."""
        layer = make_layer(w, inp, capacity_factor=args.capacity_factor)
        res = timed_layer(layer, K, W)
        routed = layer.routed.cpu().numpy().astype(np.int64)
        R = layer.T * layer.k
        dropped = int(np.maximum(routed - layer.C, 0).sum())
        out = {"capacity_factor": args.capacity_factor, "capacity": layer.C,
               "value": throughput(w.T, world, res["ms_per_step"]), "unit": UNIT,
               "ms_per_step": res["ms_per_step"],
               "padded_time_over_unpadded": res["ms_per_step"] / unpadded_ms,
               "dropped_rows": dropped, "dropped_fraction": dropped / R,
               "gemm_rows_over_routed": layer.R / R,
               "kernels_ms": res["kernels_ms"], "gpu_launches": res["launches"],
               "note": "every expert padded to C rows with zero rows, overflow dropped; same "
                       "grouped GEMM kernels on E*C rows"}
        del layer
        torch.cuda.empty_cache()
        return out

    def e2e(layer, inp, K):
        """Same step through the public API with host inputs: every step copies
        its inputs from pinned host memory and reads its outputs back
        (HostPipeline: step i+1's input copies and step i-1's output copies
        overlap step i; each step still starts from a flushed L2)."""
        T, k = layer.T, layer.k
        hin = {"x": bf16_tensor(inp["x"], "cpu").pin_memory(),
               "dY": bf16_tensor(inp["dY"], "cpu").pin_memory()}
        if not layer.learned:
            hin["idx"] = torch.from_numpy(inp["idx"]).pin_memory()
            hin["glogit"] = torch.from_numpy(inp["glogit"]).pin_memory()
        hout = {n: torch.empty(T, layer.d, dtype=torch.bfloat16).pin_memory() for n in ("out", "dX")}
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        d2h = sum(t.numel() * t.element_size() for t in hout.values())
        pipe = HostPipeline(layer, input_names=tuple(hin), output_names=tuple(hout))
        pipe.run([hin] * 2, [hout] * 2, before_step=flush.zero_)      # warm-up
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True); e = torch.cuda.Event(enable_timing=True)
        s.record()
        pipe.run([hin] * K, [hout] * K, before_step=flush.zero_)
        e.record()
        e.synchronize()
        barrier()
        ms = allmax(s.elapsed_time(e) / K, dev)
        return {"value": throughput(T, world, ms), "unit": UNIT, "ms_per_step": ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "inputs copied from pinned host memory and results copied back every "
                        "step; the copies of neighbouring steps overlap on two copy streams "
                        "(HostPipeline); the L2 flush before each step is inside the timed region"}

    w = wl.get_workload(args.workload)
    inp = wl.generate(w, seed=args.seed + rank, with_backward=True)
    main = timed(w, inp, args.steps, args.warmup, with_e2e=True)
    del inp
    cmp_res = None
    if args.compare:
        w2 = wl.get_workload(args.compare)
        inp2 = wl.generate(w2, seed=args.seed + rank, with_backward=True)
        cmp_res = timed(w2, inp2, args.steps, args.warmup, with_e2e=False, sample_clocks=False)
        cmp_res["workload"] = w2.name
        del inp2

    skew_res = None
    if args.skew_workload:
        w4 = wl.get_workload(args.skew_workload)
        inp4 = wl.generate(w4, seed=args.seed + rank, with_backward=True)
        skew_res = timed(w4, inp4, args.steps, args.warmup, with_e2e=False, sample_clocks=False)
        skew_res["workload"] = w4.name
        del inp4

    mx_res = None
    if args.mxfp8_workload:
        w3 = wl.get_workload(args.mxfp8_workload)
        inp3 = wl.generate(w3, seed=args.seed + rank, with_backward=True)
        layer = make_layer(w3, inp3, mxfp8=True)
        del inp3
        bf = timed_layer(layer, args.steps, args.warmup)
        mx = timed_layer(layer, args.steps, args.warmup,
                         step=lambda mark=None: layer.step_mxfp8(mark, requantize=True))
        mxc = timed_layer(layer, args.steps, args.warmup,
                          step=lambda mark=None: layer.step_mxfp8(mark, requantize=False))
        # Xp and A kept between forward and backward only as MXFP8 codes + scales
        mxs = timed_layer(layer, args.steps, args.warmup,
                          step=lambda mark=None: layer.step_mxfp8(mark, requantize=False,
                                                                  saved="mxfp8"))
        mxs["activation_bytes"] = layer.activation_bytes()
        # the dgrad GEMM in MXFP8 as well (weights cached, dh1/dh3 quantised in the step)
        mxd = timed_layer(layer, args.steps, args.warmup,
                          step=lambda mark=None: layer.step_mxfp8(mark, requantize=False,
                                                                  dgrad="mxfp8"))
        del layer
        torch.cuda.empty_cache()
        mx_res = (w3, bf, mx, mxc, mxs, mxd)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    ms = main["ms_per_step"]
    value = throughput(w.T, world, ms)
    km = main["kernels_ms"]
    flops, bytes_ = work_per_launch(w)
    # the dominant kernel: the single-kernel call with the largest share of the
    # step, among the calls on the step's own stream
    single = {k: v for k, v in km.items()
              if (k in flops or k in bytes_) and k not in main["side_labels"]}
    dom = max(single, key=single.get)
    traffic = None
    try:
        with open(PROFILE_TRAFFIC) as f:
            prof = json.load(f).get(dom)
        kind = "gemm" if dom in flops else "rows"
        if prof and prof.get("src_sha") == sources_sha(kind) and prof.get("workload") == w.key:
            traffic = prof["dram_bytes_per_launch"]
    except (OSError, ValueError):
        pass
    # The timed region is tens of milliseconds at full SM clock (see "clocks"),
    # so the tensor-bound kernels are measured against the burst cuBLAS peak;
    # the sustained one (seconds-long loop under the power cap, lower clock)
    # is reported beside it.
    sm_mhz = (main.get("clocks") or {}).get("sm_mhz")
    burst, sustained = peaks["bf16_tflops"], peaks["bf16_tflops_sustained"]
    if dom in flops:
        ach = flops[dom] / (km[dom] / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": burst, "unit": "TFLOP/s",
                "frac": ach / burst, "traffic": traffic,
                "algorithmic_flops_per_launch": flops[dom],
                "frac_of_sustained": ach / sustained, "sm_mhz_median": sm_mhz,
                "peak_note": f"{peaks['source']} cuBLAS bf16, burst (sustained {sustained:.1f} "
                             f"TFLOP/s reported as frac_of_sustained)"}
    else:
        ach = bytes_[dom] / (km[dom] / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": traffic,
                "algorithmic_bytes_per_launch": bytes_[dom],
                "peak_note": f"{peaks['source']} copy bandwidth"}
    gemm_labels = [k for k in flops if k in km]
    gemm_ms = sum(km[k] for k in gemm_labels)
    gemm_tflops = sum(flops[k] for k in gemm_labels) / (gemm_ms / 1e3) / 1e12
    rows = {k: {"ms": km[k], "GB_s": bytes_[k] / (km[k] / 1e3) / 1e9,
                "frac_hbm": bytes_[k] / (km[k] / 1e3) / 1e9 / peaks["hbm_gbs"]}
            for k in bytes_ if k in km}
    for k, ms_alone in main.get("alone_ms", {}).items():
        # run beside the wgrad GEMM on the layer's second stream: its time
        # there is shared; its bandwidth is that of the call timed by itself
        gbs = bytes_[k] / (ms_alone / 1e3) / 1e9
        rows[k] = {"ms": ms_alone, "GB_s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                   "ms_beside_gemm_wgrad": km.get(k), "timed": "alone, L2 flushed"}
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded normals (x, W, dY), uniform random top-4 routing",
        "config": {"workload": w.name, "key": w.key, "T": w.T, "d": w.d, "E": w.E, "k": w.k,
                   "h": w.h, "routing": w.routing, "tokens_per_gpu": w.T,
                   "l2": "flushed between timed steps (256 MB write, twice the L2)",
                   "parallelism": f"{world} replica(s), token-sharded, no data-path collective"},
        "roofline": roof,
        "gemm": {"tflops": gemm_tflops, "frac_of_peak": gemm_tflops / burst,
                 "frac_of_sustained": gemm_tflops / sustained, "ms": gemm_ms,
                 "peak": burst, "peak_note": "burst cuBLAS bf16", "sm_mhz_median": sm_mhz,
                 # each grouped GEMM against the same burst bf16 peak
                 "per_kernel": {k: {"ms": km[k], "tflops": flops[k] / (km[k] / 1e3) / 1e12,
                                    "frac_of_peak": flops[k] / (km[k] / 1e3) / 1e12 / burst}
                                for k in gemm_labels}},
        "dispatch_gbs": rows.get("dispatch", {}).get("GB_s"),
        "row_kernels": rows,
        "kernels_ms": km,
        "e2e": main["e2e"],
        "gpu_launches": main["launches"],
        "clocks": main["clocks"],
        "row_tile_overhead": main["row_tile_overhead"],
    }
    if "padded" in main:
        out["padded"] = main["padded"]
    rec = main["recompute"]
    out["recompute"] = {
        "value": throughput(w.T, world, rec["ms_per_step"]), "unit": UNIT,
        "ms_per_step": rec["ms_per_step"], "ratio_to_main": ms / rec["ms_per_step"],
        "activation_bytes_kept": rec["activation_bytes"],
        "extra_ms": {k: rec["kernels_ms"][k] for k in ("dispatch_recompute", "gemm_up_recompute")},
        "note": "backward gathers Xp from x again and recomputes H1/H3/A; only x, routing and Yp "
                "live from forward to backward"}
    if cmp_res is not None:
        cv = world * wl.get_workload(args.compare).T / (cmp_res["ms_per_step"] / 1e3)
        out["compare"] = {"workload": cmp_res["workload"], "value": cv, "unit": UNIT,
                          "ms_per_step": cmp_res["ms_per_step"], "ratio_to_main": cv / value,
                          "kernels_ms": cmp_res["kernels_ms"], "gpu_launches": cmp_res["launches"],
                          "row_tile_overhead": cmp_res["row_tile_overhead"],
                          "padded": cmp_res.get("padded")}
    if skew_res is not None:
        sv = world * wl.get_workload(args.skew_workload).T / (skew_res["ms_per_step"] / 1e3)
        out["skew"] = {"workload": skew_res["workload"], "value": sv, "unit": UNIT,
                       "ms_per_step": skew_res["ms_per_step"], "ratio_to_main": sv / value,
                       "kernels_ms": skew_res["kernels_ms"], "gpu_launches": skew_res["launches"],
                       "row_tile_overhead": skew_res["row_tile_overhead"],
                       "padded": skew_res.get("padded"),
                       "note": "learned router x W_r + b with a Zipf(1.2) expert bias (seed 0: 100 of 128 "
                               "experts empty, the hottest holds a quarter of the routed rows); "
                               "the step includes the fp32 router GEMM and its backward"}
    if mx_res is not None:
        w3, bf, mx, mxc, mxs, mxd = mx_res
        fl, _ = work_per_launch(w3)
        fwd_flops = fl["gemm_up"] + fl["gemm_down"]
        bf_fwd = bf["kernels_ms"]["gemm_up"] + bf["kernels_ms"]["gemm_down"]
        mx_fwd = mx["kernels_ms"]["gemm_fwd_mxfp8"]
        out["mxfp8"] = {
            "workload": w3.name,
            "bf16": {"value": world * w3.T / (bf["ms_per_step"] / 1e3), "ms_per_step": bf["ms_per_step"],
                     "fwd_gemm_ms": bf_fwd, "fwd_gemm_tflops": fwd_flops / (bf_fwd / 1e3) / 1e12},
            "mxfp8_fwd": {"value": world * w3.T / (mx["ms_per_step"] / 1e3), "ms_per_step": mx["ms_per_step"],
                          "fwd_gemm_ms": mx_fwd, "fwd_gemm_tflops": fwd_flops / (mx_fwd / 1e3) / 1e12,
                          "weight_quantize_ms": mx["kernels_ms"].get("mx_quantize_weights")},
            "mxfp8_fwd_cached_weights": {
                "value": world * w3.T / (mxc["ms_per_step"] / 1e3), "ms_per_step": mxc["ms_per_step"],
                "note": "weights re-quantised once per optimizer step, outside the step"},
            "mxfp8_fwd_cached_weights_mxfp8_saved": {
                "value": world * w3.T / (mxs["ms_per_step"] / 1e3), "ms_per_step": mxs["ms_per_step"],
                "dequantize_ms": mxs["kernels_ms"].get("mx_dequantize_saved"),
                "activation_bytes_kept": {k: mxs["activation_bytes"][k] for k in ("saved", "mxfp8_saved")},
                "note": "Xp and A kept between forward and backward as E4M3 codes + E8M0 scales "
                        "(no bf16 copy written in the forward), dequantised to bf16 before the backward"},
            "mxfp8_fwd_and_dgrad_cached_weights": {
                "value": world * w3.T / (mxd["ms_per_step"] / 1e3), "ms_per_step": mxd["ms_per_step"],
                "dgrad_gemm_ms": mxd["kernels_ms"].get("gemm_dx_mxfp8"),
                "dact_gemm_ms": mxd["kernels_ms"].get("gemm_dact"),
                "bf16_dact_gemm_ms": bf["kernels_ms"].get("gemm_dact"),
                "bf16_dgrad_gemm_ms": bf["kernels_ms"].get("gemm_dx"),
                "dgrad_gemm_speedup": bf["kernels_ms"]["gemm_dx"] / mxd["kernels_ms"]["gemm_dx_mxfp8"],
                "note": "dh1/dh3 quantised along h in the dact GEMM's epilogue, W1/W3 copies "
                        "quantised along h once per optimizer step; wgrad stays bf16"},
            "step_speedup_fwd_and_dgrad_cached_weights": bf["ms_per_step"] / mxd["ms_per_step"],
            "step_speedup": bf["ms_per_step"] / mx["ms_per_step"],
            "step_speedup_cached_weights": bf["ms_per_step"] / mxc["ms_per_step"],
            "fwd_gemm_speedup": bf_fwd / mx_fwd,
            # the fp8 dense peak taken as twice the measured burst bf16 one
            # (the nominal fp8 / bf16 ratio of the part, 4.5 / 2.25 PFLOP/s)
            "fwd_gemm_frac_of_fp8_peak": fwd_flops / (mx_fwd / 1e3) / 1e12 / (2 * burst),
            "fp8_peak": 2 * burst,
            "unit": UNIT, "units_note": "fp8 GEMM TFLOP/s compare to a 2x higher tensor peak than bf16",
            "kernels_ms_mxfp8": mx["kernels_ms"],
        }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, args.seed, args.cpu_seconds)
    print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def device_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:  # noqa: BLE001
        return None


# ------------------------------------------------------------ oracle timing

def _oracle_step(w, inp, Ts):
    """fp64 oracle forward + backward on the first Ts tokens of the workload."""
    import oracle.layer as ol
    sub = dict(inp)
    for key in ("x", "dY", "idx", "glogit"):
        if key in sub:
            sub[key] = inp[key][:Ts]
    t0 = time.perf_counter()
    fwd = ol.layer_forward(sub, w.k, w.E)
    ol.layer_backward(sub, fwd, w.k, w.E)
    return time.perf_counter() - t0


def _calibrate(w, inp, seconds):
    t = _oracle_step(w, inp, 256)
    Ts = int(256 * seconds / max(t, 1e-3))
    return max(64, min(w.T, Ts))


def cpu_baseline(w, seed, seconds):
    from token_dispatch_grouped_router_gb300 import workloads as wl
    inp = wl.generate(w, seed=seed, with_backward=True)
    Ts = _calibrate(w, inp, seconds)
    dt = _oracle_step(w, inp, Ts)
    return {"value": Ts / dt, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "seconds": dt,
            "sample": f"first {Ts} of {w.T} tokens of {w.key}, full weights, fp64 numpy "
                      f"forward+backward, one pass"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from token_dispatch_grouped_router_gb300 import workloads as wl
    w = wl.get_workload(args.workload)
    inp = wl.generate(w, seed=args.seed, with_backward=True)
    per_step = args.ref_seconds / max(1, args.steps + args.warmup)   # a few minutes in total
    Ts = _calibrate(w, inp, per_step)
    for _ in range(args.warmup):
        _oracle_step(w, inp, Ts)
    times = [_oracle_step(w, inp, Ts) for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    value = Ts / (ms / 1e3)
    sample = (f"first {Ts} of {w.T} tokens of {w.key} per step, full weights, fp64 numpy "
              "forward+backward")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic: seeded normals (x, W, dY), uniform random top-4 routing",
           "config": {"workload": w.name, "key": w.key, "T": w.T, "d": w.d, "E": w.E, "k": w.k,
                      "h": w.h, "routing": w.routing, "tokens_per_step": Ts},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
