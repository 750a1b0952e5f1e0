"""Seeded synthetic inputs for the FP8 delayed-scaling linear workloads.

This module only draws random numbers with fixed seeds. It holds none of the
method's arithmetic (no cast, no scale, no GEMM, no update), so the CUDA
path's tests and benchmark and the CPU oracle can both consume the same bits
without sharing any of the computation.

Shapes and distributions follow the workloads the pages describe:

* ``linear768``: one 768->768 linear with bias, input 1024x768 uniform [0, 1),
  weight and bias uniform (-1/sqrt(768), 1/sqrt(768)), seed 12345 ("Transformer
  Engine으로 FP8 사용하기", the te.Linear example under "FP8 사용방안(recipe)").
* ``linear768_drift``: the same layer over 32 steps, the input scaled by
  1.1**t at step t and a bf16 output gradient ~ N(0, 1e-3) drawn from seed
  1000 + t (exercises the amax history roll and saturation).
* ``transformer_block``: QKV 4096->12288 and proj 4096->4096 at M = 8192 tokens
  (sequence 2048 x batch 4, a multiple of 16 as the same page's "주의!" section
  asks), bf16 activations ~ N(0, 1) with 0.1 % of positions multiplied by 50,
  weights ~ N(0, 0.02), bf16 output gradient ~ N(0, 1e-3).
* ``mlp``: up 4096->14336 and down 14336->4096 at M = 16384 bf16 tokens; the up
  input ~ N(0, 1), the down input silu(a) * b with a, b ~ N(0, 1) (drawn on the
  host only to give SwiGLU-shaped values), gradients ~ N(0, 1e-4).
* ``master_step``: a flat buffer of parameters, fp32 master ~ N(0, 0.02),
  bf16 gradients ~ N(0, 1e-5) times the loss scale 2**16, with 0.01 % of the
  positions set to +-Inf / NaN (half each) on the step that injects them
  ("LLM) Mixed-Precision 개념 및 학습 방법 알아보기", the dynamic loss-scaling
  procedure).

N(0, s) means standard deviation s. Every generator takes a ``device``: on the
CPU it uses a CPU ``torch.Generator``; for full-size GPU runs it uses a CUDA
generator (different bits, same distribution) and the caller copies the bits
to the host for the oracle. Parity never depends on the two generators
agreeing.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "gen",
    "linear768",
    "linear768_drift_step",
    "transformer_block",
    "mlp",
    "master_step",
    "uniform",
    "normal",
]


def gen(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def uniform(shape, lo: float, hi: float, g: torch.Generator, dtype=torch.float32, device="cpu"):
    t = torch.rand(shape, generator=g, dtype=torch.float32, device=device)
    return (t * (hi - lo) + lo).to(dtype)


def normal(shape, std: float, g: torch.Generator, dtype=torch.float32, device="cpu"):
    t = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    return (t * std).to(dtype)


@dataclass
class Linear768:
    x: torch.Tensor      # (1024, 768) fp32, U[0, 1)
    w: torch.Tensor      # (768, 768) fp32, U(-1/sqrt(768), 1/sqrt(768))
    b: torch.Tensor      # (768,) fp32, same range


def linear768(seed: int = 12345, device="cpu") -> Linear768:
    g = gen(seed, device)
    bound = 1.0 / math.sqrt(768.0)
    x = torch.rand((1024, 768), generator=g, dtype=torch.float32, device=device)
    w = uniform((768, 768), -bound, bound, g, device=device)
    b = uniform((768,), -bound, bound, g, device=device)
    return Linear768(x=x, w=w, b=b)


def linear768_drift_step(base: Linear768, t: int, device="cpu"):
    """Inputs of step t of the 32-step drift run: (x_t fp32, dy_t bf16)."""
    x_t = (base.x.to(device) * (1.1 ** t)).to(torch.float32)
    dy_t = normal((1024, 768), 1e-3, gen(1000 + t, device), dtype=torch.bfloat16, device=device)
    return x_t, dy_t


@dataclass
class TransformerBlock:
    x: torch.Tensor       # (M, 4096) bf16
    w_qkv: torch.Tensor   # (12288, 4096) bf16
    w_proj: torch.Tensor  # (4096, 4096) bf16
    dy_qkv: torch.Tensor  # (M, 12288) bf16
    dy_proj: torch.Tensor  # (M, 4096) bf16


def transformer_block(seed: int = 3, m: int = 8192, d: int = 4096, device="cpu",
                      outlier_frac: float = 1e-3, outlier_mult: float = 50.0) -> TransformerBlock:
    g = gen(seed, device)
    x = torch.randn((m, d), generator=g, dtype=torch.float32, device=device)
    k = max(1, int(round(outlier_frac * x.numel())))
    pos = torch.randint(0, x.numel(), (k,), generator=g, device=device)
    x.view(-1)[pos] *= outlier_mult
    x = x.to(torch.bfloat16)
    w_qkv = normal((3 * d, d), 0.02, g, torch.bfloat16, device)
    w_proj = normal((d, d), 0.02, g, torch.bfloat16, device)
    dy_qkv = normal((m, 3 * d), 1e-3, g, torch.bfloat16, device)
    dy_proj = normal((m, d), 1e-3, g, torch.bfloat16, device)
    return TransformerBlock(x=x, w_qkv=w_qkv, w_proj=w_proj, dy_qkv=dy_qkv, dy_proj=dy_proj)


@dataclass
class MLP:
    x_up: torch.Tensor    # (M, 4096) bf16
    x_down: torch.Tensor  # (M, 14336) bf16, silu(a) * b
    w_up: torch.Tensor    # (14336, 4096) bf16
    w_down: torch.Tensor  # (4096, 14336) bf16


def mlp(seed: int = 4, m: int = 16384, d: int = 4096, h: int = 14336, device="cpu") -> MLP:
    g = gen(seed, device)
    x_up = torch.randn((m, d), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)
    a = torch.randn((m, h), generator=g, dtype=torch.float32, device=device)
    b = torch.randn((m, h), generator=g, dtype=torch.float32, device=device)
    x_down = (torch.nn.functional.silu(a) * b).to(torch.bfloat16)
    del a, b
    w_up = normal((h, d), 0.02, g, torch.bfloat16, device)
    w_down = normal((d, h), 0.02, g, torch.bfloat16, device)
    return MLP(x_up=x_up, x_down=x_down, w_up=w_up, w_down=w_down)


def mlp_grad(step: int, which: int, m: int, n: int, seed: int = 4, device="cpu") -> torch.Tensor:
    """bf16 output gradient ~ N(0, 1e-4) of shape (m, n) for step ``step``.

    ``which`` is 0 for the up projection's output gradient, 1 for the down's.
    """
    return normal((m, n), 1e-4, gen(1000 * seed + 2 * step + which, device),
                  torch.bfloat16, device)


def master_weights(n: int, seed: int = 5, device="cpu") -> torch.Tensor:
    return normal((n,), 0.02, gen(seed, device), torch.float32, device)


def master_step(n: int, step: int, seed: int = 5, loss_scale: float = 2.0 ** 16,
                inject: bool = False, inject_frac: float = 1e-4, device="cpu") -> torch.Tensor:
    """bf16 gradients of one step: N(0, 1e-5) * loss_scale, optional +-Inf/NaN."""
    g = gen(seed * 1000 + 17 + step, device)
    grad = (torch.randn((n,), generator=g, dtype=torch.float32, device=device)
            * (1e-5 * loss_scale)).to(torch.bfloat16)
    if inject and n > 0:
        k = max(1, int(round(inject_frac * n)))
        pos = torch.randint(0, n, (k,), generator=g, device=device)
        half = k // 2
        vals = torch.empty((k,), dtype=torch.float32, device=device)
        vals[:half] = float("nan")
        sign = torch.where(torch.rand((k - half,), generator=g, device=device) < 0.5, -1.0, 1.0)
        vals[half:] = sign * float("inf")
        grad[pos] = vals.to(torch.bfloat16)
    return grad


# Bit views shared by both sides (no arithmetic).
def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    """uint16 bit pattern of a bf16 tensor, as an int16 CPU tensor view."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16)
