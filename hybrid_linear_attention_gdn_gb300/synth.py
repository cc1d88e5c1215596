"""Seeded synthetic inputs for the GDN slot-pool step.

This module only draws random numbers; it contains none of the method's
arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Recipe (the value distributions of the Qwen3.5-shaped GDN layer workloads;
variances are read as variances, so N(0, 0.25) means std 0.5):

* q/k/v activations entering the conv:   N(0, 1)
* a, b (gate pre-activations):           N(0, 1)
* A_log:                                 U(0, ln 16)
* dt_bias:                               0
* conv1d weights [C][W]:                 N(0, 0.25)
* initial ssm state and conv history:    N(0, 0.1)
* slot ids:                              a random permutation of the pool

Everything is drawn in fp32 on the CPU from ``torch.Generator`` seeded with the
workload's seed and rounded (RNE) to bf16 where the workload is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class LayerShape:
    """Shape of one GDN layer and its state pool."""

    name: str
    hk: int          # QK heads
    hv: int          # V heads (GQA: V head h reads QK head h // (hv // hk))
    dk: int
    dv: int
    w: int           # conv width
    num_slots: int
    act: str         # dtype of qkv / a / b / out: "f32" | "bf16"
    conv: str        # dtype of the conv history: "f32" | "bf16"

    @property
    def channels(self) -> int:
        return 2 * self.hk * self.dk + self.hv * self.dv

    @property
    def act_dtype(self) -> torch.dtype:
        return _DT[self.act]

    @property
    def conv_dtype(self) -> torch.dtype:
        return _DT[self.conv]

    def replace(self, **kw) -> "LayerShape":
        d = dict(self.__dict__)
        d.update(kw)
        return LayerShape(**d)


# Tiny GDN decode: 2 QK heads, 4 V heads, dk=dv=16, width 4, fp32, 8 slots.
TINY = LayerShape("tiny_gdn_h2x4_d16", 2, 4, 16, 16, 4, 8, "f32", "f32")
# Qwen3.5-shaped GDN layer: 16 QK heads, 32 V heads, dk=dv=128, width 4 over
# 8192 channels, bf16 activations and conv history, fp32 state, 512 slots.
QWEN = LayerShape("qwen35_gdn_h16x32_d128", 16, 32, 128, 128, 4, 512, "bf16", "bf16")


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, gen: torch.Generator, dtype=torch.float32) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32) * std
    return x.to(dtype)


def params(shape: LayerShape, gen: torch.Generator):
    """(conv_w [C][W] fp32, A_log [HV] fp32, dt_bias [HV] fp32)."""
    conv_w = normal((shape.channels, shape.w), 0.5, gen)
    A_log = torch.rand((shape.hv,), generator=gen, dtype=torch.float32) * math.log(16.0)
    dt_bias = torch.zeros((shape.hv,), dtype=torch.float32)
    return conv_w, A_log, dt_bias


def pool(shape: LayerShape, gen: torch.Generator, num_slots: int | None = None):
    """(ssm [N][HV][DV][DK] fp32, conv [N][W-1][C] conv dtype), N(0, 0.1)."""
    n = shape.num_slots if num_slots is None else num_slots
    std = math.sqrt(0.1)
    ssm = normal((n, shape.hv, shape.dv, shape.dk), std, gen)
    conv = normal((n, shape.w - 1, shape.channels), std, gen, shape.conv_dtype)
    return ssm, conv


def tokens(shape: LayerShape, gen: torch.Generator, lead: tuple):
    """(qkv [*lead][C], a [*lead][HV], b [*lead][HV]) in the activation dtype."""
    qkv = normal(lead + (shape.channels,), 1.0, gen, shape.act_dtype)
    a = normal(lead + (shape.hv,), 1.0, gen, shape.act_dtype)
    b = normal(lead + (shape.hv,), 1.0, gen, shape.act_dtype)
    return qkv, a, b


def slot_ids(num_slots: int, n: int, gen: torch.Generator) -> torch.Tensor:
    """n distinct slot ids drawn from [0, num_slots)."""
    return torch.randperm(num_slots, generator=gen)[:n].to(torch.int32)


def accept_lengths(B: int, T: int, gen: torch.Generator) -> torch.Tensor:
    """Accepted draft count per request, uniform in 1..T."""
    return torch.randint(1, T + 1, (B,), generator=gen, dtype=torch.int32)
