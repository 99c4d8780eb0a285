"""Python binding of include/polar.h (Polar Express orthogonalisation), argument marshalling only.

The kernels live in the same library as the attention (libswa_attn.so); this module reuses its loaded
handle and raises at import if the library is missing. Every computation runs in the library's CUDA
kernels.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from .attn import ATTN_OK, AttnError, lib

EXPORTED = ("pe_workspace_bytes", "pe_step_flops", "pe_normalize", "pe_step", "polar_express")

_c = ctypes
lib.pe_workspace_bytes.argtypes = [_c.c_int, _c.c_int, _c.c_int]
lib.pe_workspace_bytes.restype = _c.c_size_t
lib.pe_step_flops.argtypes = [_c.c_int, _c.c_int, _c.c_int]
lib.pe_step_flops.restype = _c.c_double
lib.pe_normalize.argtypes = [_c.c_void_p, _c.c_void_p] + [_c.c_int] * 3 + [_c.c_void_p, _c.c_size_t, _c.c_void_p]
lib.pe_normalize.restype = _c.c_int
lib.pe_step.argtypes = [_c.c_void_p, _c.c_void_p] + [_c.c_int] * 4 + [_c.c_void_p, _c.c_size_t, _c.c_void_p]
lib.pe_step.restype = _c.c_int
lib.polar_express.argtypes = [_c.c_void_p, _c.c_void_p] + [_c.c_int] * 4 + [_c.c_void_p, _c.c_size_t, _c.c_void_p]
lib.polar_express.restype = _c.c_int


def _check(name, t, shape=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda" or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _dims(g: torch.Tensor):
    if g.dim() == 2:
        return 1, g.shape[0], g.shape[1]
    if g.dim() == 3:
        return g.shape[0], g.shape[1], g.shape[2]
    raise ValueError("expected a matrix [m, n] or a batch [batch, m, n]")


def workspace_bytes(batch: int, m: int, n: int) -> int:
    return int(lib.pe_workspace_bytes(batch, m, n))


def step_flops(batch: int, m: int, n: int) -> float:
    """FLOPs one step executes on the tensor cores on the current device (attn_init first)."""
    return float(lib.pe_step_flops(batch, m, n))


def _workspace(ws, nbytes, device):
    if ws is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if ws.dtype != torch.uint8 or not ws.is_contiguous() or ws.numel() < nbytes:
        raise ValueError(f"workspace must be a contiguous uint8 tensor of at least {nbytes} bytes")
    return ws


def _stream(s, device):
    s = s if s is not None else torch.cuda.current_stream(device)
    return _c.c_void_p(s.cuda_stream or None)


def normalize(g: torch.Tensor, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    _check("g", g)
    batch, m, n = _dims(g)
    out = torch.empty_like(g) if out is None else out
    _check("out", out, g.shape)
    nbytes = workspace_bytes(batch, m, n)
    ws = _workspace(workspace, nbytes, g.device)
    rc = lib.pe_normalize(g.data_ptr(), out.data_ptr(), batch, m, n, ws.data_ptr(), ws.numel(),
                          _stream(stream, g.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "pe_normalize")
    return out


def step(x: torch.Tensor, index: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
         stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """One step with coefficient triple `index`; returns (Y, A, B), A and B views into the workspace."""
    _check("x", x)
    batch, m, n = _dims(x)
    out = torch.empty_like(x) if out is None else out
    _check("out", out, x.shape)
    nbytes = workspace_bytes(batch, m, n)
    ws = _workspace(workspace, nbytes, x.device)
    rc = lib.pe_step(x.data_ptr(), out.data_ptr(), batch, m, n, int(index), ws.data_ptr(), ws.numel(),
                     _stream(stream, x.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "pe_step")
    s = min(m, n)
    a = ws[: batch * s * s * 2].view(torch.bfloat16).view(batch, s, s)
    b_off = (batch * s * s * 2 + 255) // 256 * 256
    b = ws[b_off: b_off + batch * s * s * 2].view(torch.bfloat16).view(batch, s, s)
    return out, a, b


def polar_express(g: torch.Tensor, steps: int = 5, out: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _check("g", g)
    batch, m, n = _dims(g)
    out = torch.empty_like(g) if out is None else out
    _check("out", out, g.shape)
    ws = _workspace(workspace, workspace_bytes(batch, m, n), g.device)
    rc = lib.polar_express(g.data_ptr(), out.data_ptr(), batch, m, n, int(steps), ws.data_ptr(), ws.numel(),
                           _stream(stream, g.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "polar_express")
    return out
