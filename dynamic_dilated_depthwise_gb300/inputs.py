"""Seeded synthetic inputs for the DDPM core (no arithmetic of the method here).

Both sides of every parity check -- the CUDA library and the CPU oracle --
receive the tensors drawn here; nothing in this module computes any part of
the method.

Distributions (the workloads of the "lartpang/DynamicConvolutionOperator"
README, "RTX 5090 结果": B=1, C=64, K=3 at 128^2 and 256^2, plus the
regression shape B=2, C=24, H=15, W=17 of "验证与基准"); the pages publish no
data set for this operator, so every input is synthetic:

  x, y, grad_out ~ N(0, 1)
  weight [3*C*K*K, C] ~ N(0, 1/C)         (variance 1/C: unit-variance taps)
  bias [3*C*K*K] ~ N(0, 0.01)             (variance 0.01, std 0.1)
  taps [B, 3*C*K*K, H, W] ~ N(0, 1/9)     (variance 1/9, std 1/3)

drawn in float32 from ``torch.Generator('cpu').manual_seed(seed)`` in the
order x, y, weight, bias, grad_out, taps, then cast to the compute dtype
(bfloat16 inputs are the rounded float32 draws).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Problem:
    """One DDPM problem size.  dilations are the three pyramid dilations."""
    B: int
    C: int
    H: int
    W: int
    K: int
    dilations: tuple = (1, 3, 5)
    name: str = field(default="", compare=False)

    @property
    def O(self) -> int:
        return 3 * self.C * self.K * self.K

    @property
    def pixels(self) -> int:
        return self.B * self.H * self.W


# The five workloads: regression shape, 128^2 inference, 256^2 training,
# K=5 at 128^2, and batch 8 at 256^2.
WORKLOADS = {
    "b2_c24_15x17_k3": Problem(2, 24, 15, 17, 3, name="b2_c24_15x17_k3"),
    "b1_c64_128x128_k3": Problem(1, 64, 128, 128, 3, name="b1_c64_128x128_k3"),
    "b1_c64_256x256_k3": Problem(1, 64, 256, 256, 3, name="b1_c64_256x256_k3"),
    "b1_c64_128x128_k5": Problem(1, 64, 128, 128, 5, name="b1_c64_128x128_k5"),
    "b8_c64_256x256_k3": Problem(8, 64, 256, 256, 3, name="b8_c64_256x256_k3"),
}
# seeds: 1000 + position in the list above
SEEDS = {name: 1000 + i for i, name in enumerate(WORKLOADS)}

_DTYPES = {"float32": torch.float32, "bfloat16": torch.bfloat16}


def make_inputs(p: Problem, seed: int, dtype: str = "float32", grad: bool = True,
                taps: bool = False) -> dict:
    """Draw the seeded inputs of problem p as CPU tensors of `dtype`.

    Returns a dict with x, y, weight, bias and (optionally) grad_out, taps.
    """
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    shp = (p.B, p.C, p.H, p.W)
    out = {}
    out["x"] = torch.randn(shp, generator=g, dtype=torch.float32)
    out["y"] = torch.randn(shp, generator=g, dtype=torch.float32)
    out["weight"] = torch.randn((p.O, p.C), generator=g, dtype=torch.float32) * (1.0 / p.C) ** 0.5
    out["bias"] = torch.randn((p.O,), generator=g, dtype=torch.float32) * 0.1
    if grad:
        out["grad_out"] = torch.randn((p.B, 4 * p.C, p.H, p.W), generator=g, dtype=torch.float32)
    if taps:
        out["taps"] = torch.randn((p.B, p.O, p.H, p.W), generator=g, dtype=torch.float32) * (1.0 / 3.0)
    t = _DTYPES[dtype]
    return {k: v.to(t).contiguous() for k, v in out.items()}


def make_integer_inputs(p: Problem, seed: int, dtype: str = "float32", grad: bool = True,
                        nonzeros_per_row: int = 2, taps: bool = False) -> dict:
    """Integer-valued inputs for bit-exact addressing checks.

    x, y, grad_out, bias (and taps) take values in {-1, 0, 1}; each weight row
    holds at most `nonzeros_per_row` entries from {-1, 1}.  Every product and
    sum the method forms is then a small integer, exact in bf16, tf32 and fp32.
    """
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    shp = (p.B, p.C, p.H, p.W)

    def tern(shape):
        return (torch.randint(0, 3, shape, generator=g) - 1).to(torch.float32)

    out = {"x": tern(shp), "y": tern(shp)}
    w = torch.zeros((p.O, p.C), dtype=torch.float32)
    cols = torch.randint(0, p.C, (p.O, nonzeros_per_row), generator=g)
    signs = (torch.randint(0, 2, (p.O, nonzeros_per_row), generator=g) * 2 - 1).to(torch.float32)
    for k in range(nonzeros_per_row):
        w[torch.arange(p.O), cols[:, k]] = signs[:, k]
    out["weight"] = w
    out["bias"] = tern((p.O,))
    if grad:
        out["grad_out"] = tern((p.B, 4 * p.C, p.H, p.W))
    if taps:
        out["taps"] = tern((p.B, p.O, p.H, p.W))
    t = _DTYPES[dtype]
    return {k: v.to(t).contiguous() for k, v in out.items()}
