"""Seeded synthetic inputs for the mHC seam, shared by the tests, the
benchmark and the smoke check.

This module holds no arithmetic of the method: it only draws random tensors
in a fixed order and shape.  Both the CPU oracle and the CUDA path receive
exactly the tensors drawn here.

Shapes and distributions follow the workloads of the vLLM pages
("Use AITER mHC for the delayed pre block" #56503: hidden size 5120,
hc_mult 4, 20 Sinkhorn iterations, tokens 1..16384, 80 seams per decode
step), with these synthetic stand-ins for the model's activations and
weights (no checkpoint or dataset is used):

  x       bf16 [T, n, C]      ~ N(0, 1) (drawn in fp32, one cast)
  fn      fp32 [2n+n^2, n*C]  ~ N(0, 0.02^2)
  bias    fp32 [2n+n^2]       ~ N(0, 0.1^2)
  pre_in  fp32 [T, n]         = sigmoid(U(-2, 2))
  norm_w  bf16 [C]            = 1 + N(0, 0.1^2)          (fold cases)
  y       bf16 [T, C]         ~ N(0, 1)                   (post cases)
  alpha   fp32 [3]            = (1, 1, 1)

Draw order on one ``torch.Generator``: x, fn, bias, pre_in, norm_w, y.
The stress variant redraws the comb rows of fn ~ N(0, 0.5^2) and the comb
bias ~ U(-30, 30), then scales 1% of the token rows by 1e3 (in fp32, before
the one bf16 cast) and zeroes a disjoint 1%.
"""
from __future__ import annotations

import torch

HIDDEN = 5120
HC_MULT = 4
SINKHORN_ITERS = 20


def _gen(seed: int, device: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def seam_inputs(T: int, *, n: int = HC_MULT, C: int = HIDDEN, seed: int = 0,
                fold: bool = False, with_y: bool = False, stress: bool = False,
                device: str = "cpu") -> dict:
    """Draw one seam's inputs.  ``device="cuda"`` draws with the CUDA
    generator (fast for large T); the same seed then gives different values
    than on the CPU, but every consumer of one call sees the same tensors."""
    g = _gen(seed, device)
    M = 2 * n + n * n
    kw = dict(generator=g, device=device)
    if stress:
        xf = torch.randn(T, n, C, dtype=torch.float32, **kw)
    else:
        xf = None
        x = torch.empty(T, n, C, dtype=torch.bfloat16, device=device)
        # draw in slabs so the fp32 temporary stays small for large T
        slab = max(1, (1 << 26) // max(1, n * C))
        for t0 in range(0, T, slab):
            t1 = min(T, t0 + slab)
            x[t0:t1] = torch.randn(t1 - t0, n, C, dtype=torch.float32, **kw).to(torch.bfloat16)
    fn = torch.randn(M, n * C, dtype=torch.float32, **kw) * 0.02
    bias = torch.randn(M, dtype=torch.float32, **kw) * 0.1
    pre_in = torch.sigmoid(torch.rand(T, n, dtype=torch.float32, **kw) * 4.0 - 2.0)
    norm_w = None
    if fold:
        norm_w = (1.0 + 0.1 * torch.randn(C, dtype=torch.float32, **kw)).to(torch.bfloat16)
    y = None
    if with_y:
        y = torch.randn(T, C, dtype=torch.float32, **kw).to(torch.bfloat16)
    if stress:
        fn[2 * n:] = torch.randn(n * n, n * C, dtype=torch.float32, **kw) * 0.5
        bias[2 * n:] = torch.rand(n * n, dtype=torch.float32, **kw) * 60.0 - 30.0
        k = max(1, T // 100) if T >= 2 else 0
        perm = torch.randperm(T, generator=g, device=device)
        big, zero = perm[:k], perm[k:2 * k]
        xf[big] *= 1e3
        xf[zero] = 0.0
        x = xf.to(torch.bfloat16)
        del xf
    alpha = torch.ones(3, dtype=torch.float32, device=device)
    return {"x": x, "pre_in": pre_in, "fn": fn, "bias": bias, "alpha": alpha,
            "norm_w": norm_w, "y": y, "n": n, "C": C, "T": T}


def chain_stub_delta(s: int, *, T: int = 4, C: int = HIDDEN, device: str = "cpu") -> torch.Tensor:
    """Fixed bf16 perturbation D_s ~ N(0, 0.01^2) [T, C] of the synthetic
    sublayer of seam ``s`` in the 80-seam decode chain (seed 5000 + s)."""
    g = _gen(5000 + s, device)
    return (torch.randn(T, C, dtype=torch.float32, generator=g, device=device) * 0.01).to(torch.bfloat16)


def chain_seam_params(s: int, *, n: int = HC_MULT, C: int = HIDDEN,
                      device: str = "cpu") -> dict:
    """Per-seam weights of the decode chain: seam ``s`` draws fn, bias and
    norm_w from seed 1000 + s (same distributions as ``seam_inputs``)."""
    g = _gen(1000 + s, device)
    M = 2 * n + n * n
    kw = dict(generator=g, device=device)
    fn = torch.randn(M, n * C, dtype=torch.float32, **kw) * 0.02
    bias = torch.randn(M, dtype=torch.float32, **kw) * 0.1
    norm_w = (1.0 + 0.1 * torch.randn(C, dtype=torch.float32, **kw)).to(torch.bfloat16)
    alpha = torch.ones(3, dtype=torch.float32, device=device)
    return {"fn": fn, "bias": bias, "norm_w": norm_w, "alpha": alpha}


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
