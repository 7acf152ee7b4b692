"""The arithmetic the tensor-core router relies on, checked on the CPU.

The router logits z = x W_r stay fp32-accurate on bf16 tensor cores because
(1) W_r splits exactly into three bf16 parts, W0 = RNE(W), W1 = RNE(W - W0),
W2 = RNE(W - W0 - W1), with every residual exact in fp32, and (2) the product
of two bf16 values is exact in fp32.  Both are properties of the formats (8
significant bits in bf16, 24 in fp32), checked here with torch's own
conversions over many magnitudes; the GPU kernel's output itself is compared
with the fp64 oracle in tests/test_gpu_kernels.py."""
import numpy as np
import torch


def split3(w: torch.Tensor):
    parts = []
    r = w.clone()
    for _ in range(3):
        p = r.to(torch.bfloat16)
        parts.append(p)
        r = r - p.float()                 # exact: the residual of a round to nearest
    return parts, r


def test_three_bf16_parts_reconstruct_fp32_exactly():
    rng = np.random.default_rng(0)
    mags = 2.0 ** rng.integers(-100, 100, size=20000)
    w = torch.from_numpy((rng.standard_normal(20000) * mags).astype(np.float32))
    w[:4] = torch.tensor([1.0, -3.0, 0.1, 1.0 + 2.0 ** -23])      # one bit at the bottom of the mantissa
    parts, rest = split3(w)
    assert torch.count_nonzero(rest).item() == 0
    total = sum(p.double() for p in parts)
    assert torch.equal(total, w.double())


def test_bf16_products_are_exact_in_fp32():
    rng = np.random.default_rng(1)
    a = torch.from_numpy(rng.standard_normal(50000).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy((rng.standard_normal(50000) * 1e-3).astype(np.float32)).to(torch.bfloat16)
    prod32 = a.float() * b.float()
    prod64 = a.double() * b.double()
    assert torch.equal(prod32.double(), prod64)
