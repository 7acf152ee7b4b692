"""MXFP8 codec and quantised forward of the expert FFN (fp64 CPU oracle).

TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's
CPU-baseline leg import this module; the CUDA path shares nothing with it.

Format (OLMo-core 3 tutorial, section "一个低精度格式，同时压三个地方"; "Ai2
Olmo-core 3: The Secret Behind 2.7x MoE Training Throughput", section "Boundary
Conditions of the Throughput Numbers"): elements are FP8 E4M3; every block of
32 consecutive elements along the GEMM's reduction dimension shares one E8M0
scale, a bare power of two whose exponent is read from the FP32 exponent
field.  448 is the largest E4M3 magnitude, so a block costs 32*8 + 8 bits,
8.25 bits per element.

Scale rule.  The page says the scale takes three steps, but the list of steps
is missing from the extracted text; what survives is: divide by 448, take a
power of two, and the block maximum then just fits.  Reading used here: the
block exponent e is the smallest integer with amax <= 448 * 2^e, computed
exactly from amax's binary exponent and mantissa (no rounded division),
clamped to [-127, 127]; an all-zero block gets e = -127.  The E8M0 byte is
e + 127 and the elements are RNE_E4M3(v * 2^-e), which never exceeds 448.

E4M3 encoding (OCP MX format): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
bits; exponent field 0 holds subnormals m * 2^-9; the pattern S.1111.111 is
NaN; there is no infinity; the largest finite magnitude is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

from .layer import _f64, silu

__all__ = ["E4M3_MAX", "BLOCK", "e4m3_decode", "e4m3_encode", "block_exponent",
           "quantize_blocks", "dequantize_blocks", "qdq", "expert_ffn_forward_mxfp8"]

E4M3_MAX = 448.0
BLOCK = 32


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 byte codes -> float64 values (NaN for the two NaN codes)."""
    c = np.asarray(codes).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    ex = (c >> 3) & 0xF
    man = c & 0x7
    mag = np.where(ex == 0, man * 2.0 ** -9,
                   (1.0 + man / 8.0) * np.exp2((ex - 7).astype(np.float64)))
    mag = np.where((ex == 15) & (man == 7), np.nan, mag)
    return sign * mag


# the 127 finite non-negative magnitudes, ascending with the code
_POS_VALUES = e4m3_decode(np.arange(0x7F))


def e4m3_encode(v) -> np.ndarray:
    """float64 -> E4M3 codes, round to nearest, ties to even, saturating at 448.

    Brute force over the table of finite magnitudes: the nearest value wins; on
    an exact tie the even code (mantissa LSB 0) wins.  NaN is out of contract.
    """
    v = np.asarray(v, np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("MXFP8 inputs must be finite")
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")       # first value >= a
    hi = np.minimum(hi, _POS_VALUES.size - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(_POS_VALUES[hi] == a, hi, code)           # exact hit
    # the sign is kept, also when the magnitude rounds to zero (IEEE-style)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def block_exponent(amax) -> np.ndarray:
    """Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127].

    With amax = f * 2^q (frexp, 0.5 <= f < 1) and 448 = 0.875 * 2^9, the bound
    holds for e = q - 9 exactly when f <= 0.875, otherwise e = q - 8 is the
    smallest; both comparisons are exact.
    """
    amax = np.asarray(amax, np.float64)
    f, q = np.frexp(amax)
    e = np.where(f <= 0.875, q - 9, q - 8)
    e = np.where(amax == 0, -127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize_blocks(v, axis: int = -1) -> Tuple[np.ndarray, np.ndarray]:
    """Quantise along ``axis`` in blocks of 32: returns (E4M3 codes, E8M0 bytes).

    The length along ``axis`` must be a multiple of 32.  Codes keep v's shape;
    scales have that axis divided by 32.
    """
    v = np.moveaxis(_f64(v), axis, -1)
    K = v.shape[-1]
    if K % BLOCK:
        raise ValueError("MXFP8 blocks need the reduction length to be a multiple of 32")
    blocks = v.reshape(v.shape[:-1] + (K // BLOCK, BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    e = block_exponent(amax)
    scaled = blocks * np.exp2(-e.astype(np.float64))[..., None]
    q = e4m3_encode(scaled).reshape(v.shape)
    s = (e + 127).astype(np.uint8)
    return np.moveaxis(q, -1, axis), np.moveaxis(s, -1, axis)


def dequantize_blocks(q, s, axis: int = -1) -> np.ndarray:
    q = np.moveaxis(np.asarray(q), axis, -1)
    s = np.moveaxis(np.asarray(s), axis, -1)
    vals = e4m3_decode(q)
    K = vals.shape[-1]
    scale = np.exp2(s.astype(np.float64) - 127.0)
    vals = vals.reshape(vals.shape[:-1] + (K // BLOCK, BLOCK)) * scale[..., None]
    return np.moveaxis(vals.reshape(q.shape), -1, axis)


def qdq(v, axis: int = -1) -> np.ndarray:
    """Quantise then dequantise along ``axis``."""
    q, s = quantize_blocks(v, axis)
    return dequantize_blocks(q, s, axis)


def expert_ffn_forward_mxfp8(Xp, offsets, W1, W3, W2) -> Dict[str, np.ndarray]:
    """Expert FFN forward with MXFP8 GEMM operands, fp64 arithmetic otherwise.

    Operands are quantised along each GEMM's reduction dimension: Xp along d,
    W1/W3 along d, A = silu(H1) * H3 along h, W2 along h.  Products and sums
    are exact fp64, which isolates the quantisation error from accumulation.
    """
    Xq = qdq(Xp, axis=1)
    off = np.asarray(offsets, np.int64)
    E = off.size - 1
    R = Xq.shape[0]
    h = np.asarray(W1).shape[2]
    Yp = np.zeros((R, np.asarray(W2).shape[2]))
    A = np.zeros((R, h)); H1 = np.zeros((R, h)); H3 = np.zeros((R, h))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        w1 = qdq(W1[e], axis=0)
        w3 = qdq(W3[e], axis=0)
        w2 = qdq(W2[e], axis=0)
        H1[lo:hi] = Xq[lo:hi] @ w1
        H3[lo:hi] = Xq[lo:hi] @ w3
        A[lo:hi] = silu(H1[lo:hi]) * H3[lo:hi]
        Yp[lo:hi] = qdq(A[lo:hi], axis=1) @ w2
    return {"H1": H1, "H3": H3, "A": A, "Yp": Yp}


def expert_dgrad_dx_mxfp8(dH1, dH3, offsets, W1, W3) -> np.ndarray:
    """Dgrad of the expert rows with MXFP8 GEMM operands, fp64 arithmetic
    otherwise: dXp_e = Q(dH1_e) Q(W1[e])^T + Q(dH3_e) Q(W3[e])^T.

    The reduction runs over h, so every operand is quantised along h: the
    rows of dH1 / dH3 [R, h] and the rows of W1[e] / W3[e] [d, h] (a different
    quantisation of the weights than the forward's, which runs along d).
    The same page quantises the Dgrad GEMM with the forward ones (OLMo-core 3
    tutorial, section "一个低精度格式，同时压三个地方").
    """
    off = np.asarray(offsets, np.int64)
    E = off.size - 1
    q1 = qdq(dH1, axis=1)
    q3 = qdq(dH3, axis=1)
    d = np.asarray(W1).shape[1]
    dXp = np.zeros((q1.shape[0], d))
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        dXp[lo:hi] = q1[lo:hi] @ qdq(W1[e], axis=1).T + q3[lo:hi] @ qdq(W3[e], axis=1).T
    return dXp
