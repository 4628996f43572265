"""Seeded synthetic workloads and the error metric used to compare results.

This module holds no arithmetic of the method itself: only the input
recipes (shapes, distributions, seeds) and a comparison metric.  It is the
one module that both the oracle side (tests, CPU baseline) and the CUDA side
(tests, bench) import.

Input recipe: a ``torch.Generator`` seeded with ``seed`` draws q, k, v in
that order with ``torch.randn`` in fp32 (on the CPU unless a device is
given), multiplies them by ``scale`` (1/sqrt(d) for the bf16 workloads,
1 for the fp32 one), then rounds them to the workload's dtype
(round-to-nearest-even for bf16).  The oracle receives the rounded values
widened to float64, so both sides see identical inputs.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str                 # "f32" or "bf16"
    causal: tuple              # forms to run: (True,), (False, True), ...
    scale: float
    decay: tuple | None = None  # per-head g_h, or None
    extra: dict = field(default_factory=dict)


def decay_schedule(H: int) -> tuple:
    """g_h = 1 - 2^(-5-h), h = 0..H-1 (the long-context decay workload)."""
    return tuple(1.0 - 2.0 ** (-5 - h) for h in range(H))


# The five workloads: small fp32 causal; bf16 mid-size causal and
# non-causal; bf16 long-context causal; bf16 causal with per-head decay;
# recurrent decode (256 sequences x 32 heads, state prefilled from 1024
# tokens, then 1024 single-token steps).
WORKLOADS = {
    "fp32_causal_small": Workload("fp32_causal_small", 1, 2, 512, 64, "f32",
                                  (True,), 1.0),
    "bf16_b4h16_n4096_d64": Workload("bf16_b4h16_n4096_d64", 4, 16, 4096, 64,
                                     "bf16", (True, False), 1 / math.sqrt(64)),
    "bf16_b2h16_n32768_d128": Workload("bf16_b2h16_n32768_d128", 2, 16, 32768,
                                       128, "bf16", (True,),
                                       1 / math.sqrt(128)),
    "bf16_decay_b4h8_n16384_d128": Workload(
        "bf16_decay_b4h8_n16384_d128", 4, 8, 16384, 128, "bf16", (True,),
        1 / math.sqrt(128), decay_schedule(8)),
    "decode_b256h32_d128": Workload("decode_b256h32_d128", 256, 32, 1, 128,
                                    "bf16", (True,), 1 / math.sqrt(128),
                                    extra={"prefill": 1024, "steps": 1024}),
}


def torch_dtype(name: str):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def make_qkv(B, H, N, d, dtype="bf16", scale=None, seed=0, device="cpu"):
    """q, k, v of shape [B, H, N, d], seeded, rounded to `dtype`."""
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for _ in range(3):
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32,
                        device=device)
        if scale != 1.0:
            x.mul_(scale)
        out.append(x.to(torch_dtype(dtype)))
    return tuple(out)


def make_workload_qkv(w: Workload, seed=0, device="cpu"):
    return make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.scale, seed, device)


def make_decode_tokens(B, H, d, T, dtype="bf16", scale=None, seed=0,
                       device="cpu"):
    """q, k, v for T single-token steps, each [T, B, H, d]."""
    import torch
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = []
    for _ in range(3):
        x = torch.randn((T, B, H, d), generator=g, dtype=torch.float32,
                        device=device)
        if scale != 1.0:
            x.mul_(scale)
        out.append(x.to(torch_dtype(dtype)))
    return tuple(out)


def max_row_rel_err(y, ref) -> float:
    """max over rows i of ||y_i - r_i||_inf / ||r_i||_inf (rows along the last
    axis).  Rows whose reference is exactly zero are compared absolutely."""
    y = _np64(y)
    r = _np64(ref)
    num = np.abs(y - r).max(axis=-1)
    den = np.abs(r).max(axis=-1)
    den = np.where(den > 0, den, 1.0)
    if num.size == 0:
        return 0.0
    return float((num / den).max())


def _np64(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


# tolerances (max row-relative error) by input dtype
TOL = {"f32": 1e-4, "bf16": 2e-2}
