"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the benchmark.

This module holds no attention arithmetic: it only draws q, k, v. Both sides of every
parity check read the same bf16 bits from here, so a difference between them can only come
from the computation itself.

Recipe: fp32 N(0, 1) drawn on the CPU with a `torch.Generator` seeded `seed`, in the order
q, then k, then v, each of shape [B, T, H, D], then rounded to bf16 (round to nearest even,
PyTorch's conversion). The per-layer seed of a multi-layer workload is
`1000 * config_index + layer_index`.
"""
from __future__ import annotations

import torch


def layer_seed(config_index: int, layer_index: int) -> int:
    """Seed of layer `layer_index` of workload number `config_index`."""
    return 1000 * int(config_index) + int(layer_index)


def make_qkv(B: int, T: int, H: int, D: int, seed: int, scale: float = 1.0):
    """Return (q, k, v): three CPU bf16 tensors of shape [B, T, H, D] drawn from N(0, scale^2)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    out = []
    for _ in range(3):
        x = torch.randn((B, T, H, D), generator=g, dtype=torch.float32)
        if scale != 1.0:
            x = x * scale
        out.append(x.to(torch.bfloat16))
    return tuple(out)


def bf16_bits(x: torch.Tensor):
    """The raw 16-bit patterns of a bf16 tensor as a contiguous numpy uint16 array."""
    assert x.dtype == torch.bfloat16
    return x.contiguous().view(torch.int16).numpy().view("uint16")


def from_bf16_bits(a) -> torch.Tensor:
    """Inverse of `bf16_bits`: a numpy uint16 array back to a CPU bf16 tensor."""
    import numpy as np

    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
