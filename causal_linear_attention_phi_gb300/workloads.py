"""Seeded synthetic inputs for the five workloads (shapes, distributions, seeds).

This module only draws random numbers; it holds none of the attention
arithmetic.  Both the CUDA path and the fp64 oracle consume what it produces:
the oracle takes the values after the cast to the workload's dtype (bf16 inputs
are converted exactly to fp64).

Draws use a CPU ``torch.Generator`` seeded per workload, in a fixed order
(q, k, v, dO), as fp32 N(0, 1) scaled by the stated factor and then cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    Dk: int
    Dv: int
    dtype: torch.dtype
    seed: int
    qk_scale: float = 1.0
    v_scale: float = 1.0
    do_scale: float = 1.0
    ops: tuple = field(default=("causal_fwd",))


# 1: fp32 causal forward, B=1 H=2 N=64 D=16, N(0,1), seed 0.
SMALL_F32 = Workload("causal fwd f32 B=1 H=2 N=64 Dk=Dv=16", 1, 2, 64, 16, 16,
                     torch.float32, 0, ops=("causal_fwd",))
# 2: bf16 non-causal and causal forward, B=4 H=8 N=1024 D=64, N(0,1)/sqrt(64).
FWD_BF16 = Workload("causal+noncausal fwd bf16 B=4 H=8 N=1024 Dk=Dv=64", 4, 8, 1024, 64, 64,
                    torch.bfloat16, 2, qk_scale=1 / 8, v_scale=1 / 8,
                    ops=("noncausal_fwd", "causal_fwd"))
# 5: bf16 long-context training, B=2 H=16 N=65536 D=128; Q,K ~ N(0,1)/sqrt(128); V, dO ~ N(0,1).
LONG_BF16 = Workload("causal fwd+bwd bf16 B=2 H=16 N=65536 Dk=Dv=128", 2, 16, 65536, 128, 128,
                     torch.bfloat16, 5, qk_scale=1 / math.sqrt(128), ops=("causal_fwd", "causal_bwd"))

# Retention (constant decay per head) forward at the long-context shape: B=2 H=16 N=65536 D=128 bf16;
# Q, K ~ N(0,1) * 128^-1/4 (so q . k ~ N(0,1)), V ~ N(0,1); decays from retention_gammas(16).
RETENTION_BF16 = Workload("retention fwd bf16 B=2 H=16 N=65536 Dk=Dv=128", 2, 16, 65536, 128, 128,
                          torch.bfloat16, 6, qk_scale=128 ** -0.25, ops=("retention_fwd",))


def retention_gammas(H: int) -> torch.Tensor:
    """Per-head decays (fp32 [H], CPU): 1 - gamma_h spaced evenly in log from 1/32 to 1/1024."""
    e = torch.linspace(5.0, 10.0, H, dtype=torch.float64) if H > 1 else torch.tensor([5.0], dtype=torch.float64)
    return (1.0 - torch.pow(2.0, -e)).float()


# 3: length sweep of causal fwd+bwd, bf16, B=1 H=8 D=64, N = 2^9 .. 2^16, all N(0,1).
SWEEP_NS = tuple(2 ** e for e in range(9, 17))


def sweep(N: int) -> Workload:
    return Workload("causal fwd+bwd bf16 B=1 H=8 N=%d Dk=Dv=64" % N, 1, 8, N, 64, 64,
                    torch.bfloat16, 3, ops=("causal_fwd", "causal_bwd"))


# 4: recurrent decode, fp32 state: B=64 H=8 Dk=Dv=32, 784 or 3072 steps.
@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    Dk: int
    Dv: int
    steps: int
    seed: int
    dtype: torch.dtype = torch.float32


DECODE_MNIST = DecodeWorkload("recurrent decode f32 B=64 H=8 Dk=Dv=32 steps=784", 64, 8, 32, 32, 784, 4)
DECODE_CIFAR = DecodeWorkload("recurrent decode f32 B=64 H=8 Dk=Dv=32 steps=3072", 64, 8, 32, 32, 3072, 4)


def _randn(g: torch.Generator, shape, scale: float, dtype: torch.dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def make_inputs(w: Workload, with_grad: bool = False, B: int | None = None, H: int | None = None,
                N: int | None = None):
    """Return CPU tensors (q, k, v[, dO]) of the workload's dtype and shape.

    B, H or N may be overridden (for reduced parity cases of the same recipe).
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = _randn(g, (B, H, N, w.Dk), w.qk_scale, w.dtype)
    k = _randn(g, (B, H, N, w.Dk), w.qk_scale, w.dtype)
    v = _randn(g, (B, H, N, w.Dv), w.v_scale, w.dtype)
    if not with_grad:
        return q, k, v
    dO = _randn(g, (B, H, N, w.Dv), w.do_scale, w.dtype)
    return q, k, v, dO


def make_decode_inputs(w: DecodeWorkload, steps: int | None = None):
    """Per-step q, k, v stacked as [steps, B, H, D] (CPU, fp32)."""
    T = w.steps if steps is None else steps
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = _randn(g, (T, w.B, w.H, w.Dk), 1.0, w.dtype)
    k = _randn(g, (T, w.B, w.H, w.Dk), 1.0, w.dtype)
    v = _randn(g, (T, w.B, w.H, w.Dv), 1.0, w.dtype)
    return q, k, v


def random_case(seed: int, B: int, H: int, N: int, Dk: int, Dv: int, dtype=torch.float32,
                scale: float = 1.0, with_grad: bool = False):
    """Generic seeded case for edge-case tests (same recipe, any shape)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = _randn(g, (B, H, N, Dk), scale, dtype)
    k = _randn(g, (B, H, N, Dk), scale, dtype)
    v = _randn(g, (B, H, N, Dv), 1.0, dtype)
    if not with_grad:
        return q, k, v
    dO = _randn(g, (B, H, N, Dv), 1.0, dtype)
    return q, k, v, dO
