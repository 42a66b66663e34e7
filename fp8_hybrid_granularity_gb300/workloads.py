"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random BF16 tensors and nothing else: it holds none of the
quantization or GEMM arithmetic, so both the CUDA path and the CPU oracle can
be fed the same bytes from it without sharing any of the method's code.

The recipes stand in for the data the pages train on (continual pre-training
and SFT corpora, Qwen2.5-1.5B/7B weights), which are not available here.  The
shapes are the Qwen2.5-1.5B / 7B linear-layer shapes; the distributions are
chosen to have the structure the recipe's granularity choice is about
("A Comprehensive FP8 Training Recipe ...", "What carries the argument":
activations have a wider range and strong outliers than weights).

  act_tiny : N(0, 1), 0.1% of entries multiplied by 50
  act      : z * c_k, z ~ N(0, 1), c_k ~ LogNormal(0, 1) per channel (column),
             0.1% of entries multiplied by 100
  weight   : N(0, 0.02^2)
  grad     : 1e-3 * t_3 (Student-t, 3 degrees of freedom, heavy tails)
  mx_ln    : rows [0, R/2) uniform on 1 +- 1e-3 (layer-norm-like weights),
             rows [R/2, R) N(0, 1)
  mx_ln_clamp : as mx_ln but the first half uniform on [0.990, 0.997]; after
             rounding to BF16 every value there is below 1.0 (the BF16 grid
             below 1 has spacing 2^-8), so each 32-block's amax is just under a
             power of two and most of the block clamps to the top code.  (A
             cluster at 1 +- 1e-3 rounds to exactly 1.0 in BF16: one bin, no
             clamp.)
"""
from __future__ import annotations

import zlib

import torch

KINDS = ("act_tiny", "act", "weight", "grad", "mx_ln", "mx_ln_clamp", "normal")


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF)
    return g


def make_tensor(kind: str, rows: int, cols: int, seed: int, name: str = "",
                device="cpu") -> torch.Tensor:
    """A [rows, cols] BF16 tensor drawn from ``kind`` (see module docstring).

    Generation runs in fp32 and rounds to BF16 once (round to nearest even)."""
    if kind not in KINDS:
        raise ValueError(f"unknown kind {kind!r}")
    dev = torch.device(device)
    g = _gen(seed, f"{kind}:{name}:{rows}x{cols}", dev)
    shape = (rows, cols)
    f32 = torch.float32
    if kind == "normal":
        x = torch.randn(shape, generator=g, device=dev, dtype=f32)
    elif kind == "act_tiny":
        x = torch.randn(shape, generator=g, device=dev, dtype=f32)
        hit = torch.rand(shape, generator=g, device=dev, dtype=f32) < 1e-3
        x = torch.where(hit, x * 50.0, x)
    elif kind == "act":
        z = torch.randn(shape, generator=g, device=dev, dtype=f32)
        c = torch.exp(torch.randn((1, cols), generator=g, device=dev, dtype=f32))
        x = z * c
        hit = torch.rand(shape, generator=g, device=dev, dtype=f32) < 1e-3
        x = torch.where(hit, x * 100.0, x)
    elif kind == "weight":
        x = torch.randn(shape, generator=g, device=dev, dtype=f32) * 0.02
    elif kind == "grad":
        z = torch.randn(shape, generator=g, device=dev, dtype=f32)
        chi2 = torch.zeros(shape, device=dev, dtype=f32)
        for _ in range(3):
            chi2 += torch.randn(shape, generator=g, device=dev, dtype=f32).square_()
        x = 1e-3 * z / torch.sqrt(chi2 / 3.0)
    else:  # mx_ln / mx_ln_clamp
        x = torch.randn(shape, generator=g, device=dev, dtype=f32)
        half = rows // 2
        u = torch.rand((half, cols), generator=g, device=dev, dtype=f32)
        if kind == "mx_ln":
            x[:half] = 1.0 + (2.0 * u - 1.0) * 1e-3
        else:
            x[:half] = 0.990 + u * 0.007
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a CPU BF16 tensor, as a numpy array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def from_bits(bits) -> torch.Tensor:
    """A CPU BF16 tensor from uint16 bit patterns."""
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(bits).view("int16")).view(torch.bfloat16)


# Named workloads: (tensor name, kind, rows, cols).  Sizes follow the Qwen2.5
# layer shapes: 1.5B hidden 1536, MLP 8960, QKV 2048; 7B hidden 3584, MLP 18944.
WORKLOADS = {
    "tiny_fprop": dict(seed=0, M=256, tensors=[("X", "act_tiny", 256, 512),
                                               ("W", "weight", 512, 512)]),
    "fprop_1p5b": dict(seed=1, M=8192, tensors=[
        ("X", "act", 8192, 1536), ("H", "act", 8192, 8960),
        ("W_gate", "weight", 8960, 1536), ("W_up", "weight", 8960, 1536),
        ("W_down", "weight", 1536, 8960), ("W_qkv", "weight", 2048, 1536)]),
    "linear_step_7b": dict(seed=2, M=16384, tensors=[
        ("X", "act", 16384, 3584), ("H", "act", 16384, 18944),
        ("W_gate", "weight", 18944, 3584), ("W_up", "weight", 18944, 3584),
        ("W_down", "weight", 3584, 18944),
        ("dY_gate", "grad", 16384, 18944), ("dY_up", "grad", 16384, 18944),
        ("dY_down", "grad", 16384, 3584)]),
    "mxfp8_4096": dict(seed=3, M=4096, tensors=[
        ("A", "mx_ln", 4096, 4096), ("B", "mx_ln", 4096, 4096),
        ("A_clamp", "mx_ln_clamp", 4096, 4096)]),
}


def workload_tensor(workload: str, name: str, device="cpu") -> torch.Tensor:
    spec = WORKLOADS[workload]
    for (n, kind, r, c) in spec["tensors"]:
        if n == name:
            return make_tensor(kind, r, c, spec["seed"], n, device=device)
    raise KeyError(name)
