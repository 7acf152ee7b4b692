"""Seeded synthetic inputs for the single-GPU MoE expert layer.

This module only draws random numbers and rounds them to their storage types
(bf16 bit patterns, fp32, int32).  It routes nothing, multiplies nothing and
reduces nothing, so the CUDA path and the CPU oracle can both consume its
arrays without sharing any of the layer's arithmetic.

The five workloads follow the pages' expert-pool sweep (8 -> 128 experts with
four experts per token, "Ai2 Olmo-core 3: The Secret Behind 2.7x MoE Training
Throughput", section "Measured Data on Expert Pool Scaling") and their
random-routing system benchmarks (OLMo-core 3 tutorial, section "所有 headline
数字都是随机路由下的系统基准").  The pages fix no tensor shapes, init scales or
routing recipe; the ones below are the benchmark specification's.

Random streams: ``SeedSequence(seed).spawn(9)`` gives one child per tensor, in
the fixed order x, W_r, bias permutation, W1, W3, W2, routing ids, gate
logits, dY.  A tensor that a workload does not use still consumes its child,
so every tensor's stream is independent of the others.  Normals are drawn in
fp32 and rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict
from typing import Dict, Optional

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get_workload", "generate", "bf16_bits",
           "small_workload"]


@dataclass(frozen=True)
class Workload:
    """Shape and routing recipe of one synthetic MoE-layer step."""
    key: str
    T: int            # tokens
    d: int            # model dimension
    E: int            # experts
    k: int            # experts per token
    h: int            # expert hidden dimension
    routing: str      # "learned" (x @ W_r [+ b]) or "uniform" (random ids)
    zipf: bool = False        # learned router with a Zipf(1.2) expert bias
    backward: bool = True     # the step includes the backward pass
    mxfp8: bool = False       # the workload also has an MXFP8 forward run
    seqs: int = 1             # sequences of 4096 tokens (documentation only)

    @property
    def R(self) -> int:
        """Routed rows T*k."""
        return self.T * self.k

    @property
    def name(self) -> str:
        r = "zipf-router" if self.zipf else (
            "learned-router" if self.routing == "learned" else "uniform-routing")
        return (f"moe-layer T={self.T} d={self.d} E={self.E} k={self.k} "
                f"h={self.h} {r}")

    def as_config(self) -> Dict:
        c = asdict(self)
        c["name"] = self.name
        return c


WORKLOADS: Dict[str, Workload] = {
    # tiny forward check, small enough for a full-tensor oracle comparison
    "tiny_e8": Workload("tiny_e8", T=512, d=256, E=8, k=2, h=512,
                        routing="learned", backward=False),
    # dense pool: 8 experts, 4 x 4096 tokens, forward + backward
    "dense_e8": Workload("dense_e8", T=16384, d=2048, E=8, k=4, h=1024,
                         routing="uniform", seqs=4),
    # large pool, same active size: 128 experts (~512 rows per expert)
    "pool_e128": Workload("pool_e128", T=16384, d=2048, E=128, k=4, h=1024,
                          routing="uniform", seqs=4),
    # skewed learned routing: Zipf bias, empty experts, one hot expert
    "skew_e128": Workload("skew_e128", T=16384, d=2048, E=128, k=4, h=1024,
                          routing="learned", zipf=True, seqs=4),
    # training-scale layer, 8 x 4096 tokens, BF16 and MXFP8 forward runs
    "train_e128": Workload("train_e128", T=32768, d=2048, E=128, k=4, h=1024,
                           routing="uniform", mxfp8=True, seqs=8),
}

# order of the spawned child streams
_STREAMS = ("x", "W_r", "b_perm", "W1", "W3", "W2", "idx", "glogit", "dY")


def get_workload(key: str) -> Workload:
    return WORKLOADS[key]


def small_workload(T: int, d: int, E: int, k: int, h: int,
                   routing: str = "uniform", zipf: bool = False,
                   backward: bool = True, key: str = "custom") -> Workload:
    """A workload with arbitrary (small) sizes, same recipe as the named ones."""
    return Workload(key, T=T, d=d, E=E, k=k, h=h, routing=routing, zipf=zipf,
                    backward=backward)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest-even) and return the uint16 bit patterns.

    Inputs are finite normals, so the carry into the exponent is the only
    special case and the integer add handles it.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _normal(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def generate(w: Workload, seed: int = 0, with_backward: Optional[bool] = None
             ) -> Dict[str, np.ndarray]:
    """Draw one step's inputs for workload ``w``.

    Returns a dict of numpy arrays (bf16 tensors as uint16 bit patterns):
      x[T,d] bf16, W1[E,d,h] bf16, W3[E,d,h] bf16, W2[E,h,d] bf16,
      learned routing: W_r[d,E] f32 (N(0,1/d)) and b[E] f32 (Zipf) or absent,
      uniform routing: idx[T,k] i32 (k distinct experts per token, uniform)
                       and glogit[T,k] f32 (N(0,1) gate logits),
      dY[T,d] bf16 when the step has a backward pass.
    """
    if with_backward is None:
        with_backward = w.backward
    ss = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    rng = {n: np.random.default_rng(s) for n, s in zip(_STREAMS, ss)}
    T, d, E, k, h = w.T, w.d, w.E, w.k, w.h
    out: Dict[str, np.ndarray] = {}
    out["x"] = bf16_bits(_normal(rng["x"], (T, d), 1.0))
    if w.routing == "learned":
        out["W_r"] = _normal(rng["W_r"], (d, E), 1.0 / np.sqrt(d))
        if w.zipf:
            # expert e gets Zipf rank perm[e]+1; bias 2*ln p(rank), p(r) ~ r^-1.2
            perm = rng["b_perm"].permutation(E)
            p = (perm + 1.0) ** -1.2
            p /= p.sum()
            out["b"] = (2.0 * np.log(p)).astype(np.float32)
    elif w.routing == "uniform":
        # k distinct experts per token, uniformly at random: the first k of a
        # random permutation of the E experts (drawn as argsort of uniforms)
        u = rng["idx"].random((T, E))
        out["idx"] = np.argsort(u, axis=1, kind="stable")[:, :k].astype(np.int32)
        out["glogit"] = rng["glogit"].standard_normal((T, k), dtype=np.float32)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    out["W1"] = bf16_bits(_normal(rng["W1"], (E, d, h), 1.0 / np.sqrt(d)))
    out["W3"] = bf16_bits(_normal(rng["W3"], (E, d, h), 1.0 / np.sqrt(d)))
    out["W2"] = bf16_bits(_normal(rng["W2"], (E, h, d), 1.0 / np.sqrt(h)))
    if with_backward:
        out["dY"] = bf16_bits(_normal(rng["dY"], (T, d), 1.0))
    return out
