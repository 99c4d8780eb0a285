"""Python binding of the C ABI in include/attn.h (libswa_attn.so), argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module only checks
tensor properties, passes raw device pointers and the current CUDA stream, and turns status
codes into exceptions. There is no fallback: if the library is missing, importing this module
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libswa_attn.so")

ATTN_OK = 0
ATTN_ERR_NOT_INITIALIZED = -1
ATTN_ERR_INVALID_ARG = -2
ATTN_ERR_UNSUPPORTED = -3
ATTN_ERR_CUDA = -4
ATTN_ERR_DEVICE_TIMEOUT = -5
ATTN_ERR_NO_DEVICE = -6
ATTN_ERR_SCRATCH_LIMIT = -7

EXPORTED = ("attn_init", "attn_fwd", "attn_destroy", "attn_status_string", "attn_device_status",
            "attn_selftest_wait_timeout", "attn_fwd_noalloc", "attn_fwd_kernel", "attn_fwd_gqa",
            "attn_noalloc_status", "attn_noalloc_selftest_wait_timeout", "attn_bwd_workspace_bytes", "attn_bwd",
            "attn_fwd_ve", "attn_fwd_ve_workspace_bytes")


class AttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA attention library not built: {LIB_PATH} is missing "
                          "(run __graft_entry__.build() or sliding_window_attention_04_b300/csrc/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    c_int, c_float, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    lib.attn_init.argtypes = [c_int]
    lib.attn_init.restype = c_int
    lib.attn_fwd.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                             c_int, c_int, c_float, c_float, c_void_p]
    lib.attn_fwd.restype = c_int
    lib.attn_fwd_gqa.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int,
                                 c_int, c_int, c_int, c_float, c_float, c_void_p]
    lib.attn_fwd_gqa.restype = c_int
    lib.attn_destroy.argtypes = []
    lib.attn_destroy.restype = None
    lib.attn_status_string.argtypes = [c_int]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_device_status.argtypes = []
    lib.attn_device_status.restype = c_int
    lib.attn_selftest_wait_timeout.argtypes = [c_void_p]
    lib.attn_selftest_wait_timeout.restype = c_int
    lib.attn_fwd_noalloc.argtypes = list(lib.attn_fwd.argtypes)
    lib.attn_fwd_noalloc.restype = c_int
    lib.attn_fwd_kernel.argtypes = [c_int]
    lib.attn_fwd_kernel.restype = c_int
    lib.attn_noalloc_status.argtypes = [c_void_p]
    lib.attn_noalloc_status.restype = c_int
    lib.attn_noalloc_selftest_wait_timeout.argtypes = [c_void_p]
    lib.attn_noalloc_selftest_wait_timeout.restype = c_int
    lib.attn_bwd_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int]
    lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_bwd.argtypes = [c_void_p] * 10 + [ctypes.c_size_t] + [c_int] * 7 + [c_float, c_float, c_void_p]
    lib.attn_bwd.restype = c_int
    lib.attn_fwd_ve.argtypes = ([c_void_p] * 5 + [c_int] + [c_void_p] * 4 + [ctypes.c_size_t] + [c_int] * 7 +
                                [c_float, c_float, c_void_p])
    lib.attn_fwd_ve.restype = c_int
    lib.attn_fwd_ve_workspace_bytes.argtypes = [c_int, c_int, c_int]
    lib.attn_fwd_ve_workspace_bytes.restype = ctypes.c_size_t
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.attn_status_string(int(code)).decode()


def attn_init(device: int = 0) -> None:
    rc = lib.attn_init(int(device))
    if rc != ATTN_OK:
        raise AttnError(rc, f"attn_init({device})")


def attn_destroy() -> None:
    lib.attn_destroy()


def attn_device_status() -> int:
    """Synchronise, read and clear the device error word; returns the status code."""
    return int(lib.attn_device_status())


def attn_fwd_kernel(D: int) -> str:
    """Name of the kernel attn_fwd launches for head dimension D ("ws" or "simple")."""
    rc = int(lib.attn_fwd_kernel(int(D)))
    if rc < 0:
        raise AttnError(rc, f"attn_fwd_kernel({D})")
    return "ws" if rc == 1 else "simple"


def attn_selftest_wait_timeout(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch the bounded-wait self test (see include/attn.h); check with attn_device_status()."""
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = int(lib.attn_selftest_wait_timeout(ctypes.c_void_p(s.cuda_stream or None)))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_selftest_wait_timeout")


def attn_fwd_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, lse_ptr: Optional[int], B: int, H: int, T: int,
                 D: int, window: int, causal: int, rope_base: float, eps: float, stream: Optional[int]) -> int:
    """Direct pass-through of the C call (pointers as integers); returns the status code."""
    return int(lib.attn_fwd(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                            ctypes.c_void_p(out_ptr), ctypes.c_void_p(lse_ptr or None), int(B), int(H), int(T),
                            int(D), int(window), int(causal), float(rope_base), float(eps),
                            ctypes.c_void_p(stream or None)))


def attn_fwd_gqa_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, lse_ptr: Optional[int], B: int, H: int,
                     H_kv: int, T: int, D: int, window: int, causal: int, rope_base: float, eps: float,
                     stream: Optional[int]) -> int:
    """Pass-through of the grouped-K/V-head C call (k, v have H_kv heads); returns the status code."""
    return int(lib.attn_fwd_gqa(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                ctypes.c_void_p(out_ptr), ctypes.c_void_p(lse_ptr or None), int(B), int(H),
                                int(H_kv), int(T), int(D), int(window), int(causal), float(rope_base), float(eps),
                                ctypes.c_void_p(stream or None)))


def attn_fwd_noalloc_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, lse_ptr: Optional[int], B: int, H: int,
                         T: int, D: int, window: int, causal: int, rope_base: float, eps: float,
                         stream: Optional[int]) -> int:
    """Pass-through of the allocation-free C call (see include/attn.h); returns the status code.

    For callers that must not allocate device memory: the library keeps what it needs in a
    fixed device array instead, so the only memory involved is the caller's own tensors."""
    return int(lib.attn_fwd_noalloc(ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
                                    ctypes.c_void_p(out_ptr), ctypes.c_void_p(lse_ptr or None), int(B), int(H),
                                    int(T), int(D), int(window), int(causal), float(rope_base), float(eps),
                                    ctypes.c_void_p(stream or None)))


def attn_noalloc_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Read and clear attn_fwd_noalloc's error word (waits for `stream`); returns the status code."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(lib.attn_noalloc_status(ctypes.c_void_p(s.cuda_stream or None)))


def attn_noalloc_selftest_wait_timeout(stream: Optional[torch.cuda.Stream] = None) -> int:
    """The bounded-wait self test on attn_fwd_noalloc's error word; returns the status code of the launch."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(lib.attn_noalloc_selftest_wait_timeout(ctypes.c_void_p(s.cuda_stream or None)))


def _check_input(name: str, t: torch.Tensor, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16 (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int = -1, causal: bool = True,
             rope_base: float = 10000.0, eps: float = 1e-6, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, return_lse: bool = True,
             stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Attention forward on bf16 CUDA tensors: q [B, T, H, D]; k, v [B, T, H_kv, D] with H a multiple
    of H_kv (grouped K/V heads, query head h reads K/V head h // (H // H_kv); H_kv = H is
    multi-head attention). Returns (out [B, T, H, D], lse [B, H, T] fp32 or None).

    The call is asynchronous on `stream` (default: the current stream of q's device).
    """
    _check_input("q", q)
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, D]")
    B, T, H, D = q.shape
    _check_input("k", k)
    if k.dim() != 4 or k.shape[0] != B or k.shape[1] != T or k.shape[3] != D:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [B, T, H_kv, D] = [{B}, {T}, H_kv, {D}]")
    H_kv = k.shape[2]
    if H_kv < 1 or H % H_kv != 0:
        raise ValueError(f"H = {H} is not a multiple of H_kv = {H_kv}")
    _check_input("v", v, k.shape)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_input("out", out, q.shape)
    if lse is None and return_lse:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    if lse is not None:
        if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, T):
            raise ValueError("lse must be a contiguous float32 [B, H, T] tensor")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    lse_ptr = lse.data_ptr() if lse is not None else None
    if H_kv == H:
        rc = attn_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, T, D,
                          int(window), int(bool(causal)), float(rope_base), float(eps), s.cuda_stream)
    else:
        rc = attn_fwd_gqa_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, H, H_kv, T, D,
                              int(window), int(bool(causal)), float(rope_base), float(eps), s.cuda_stream)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd" if H_kv == H else "attn_fwd_gqa")
    return out, lse


def attn_fwd_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, **kwargs):
    """attn_fwd with grouped K/V heads (k, v: [B, T, H_kv, D]); the same call as attn_fwd, which
    accepts both shapes."""
    return attn_fwd(q, k, v, **kwargs)


def attn_bwd_workspace_bytes(B: int, H: int, H_kv: int, T: int, D: int) -> int:
    return int(lib.attn_bwd_workspace_bytes(B, H, H_kv, T, D))


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
             eps: float = 1e-6, workspace: Optional[torch.Tensor] = None, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Gradients (dq [B, T, H, D], dk, dv [B, T, H_kv, D], fp32) of sum(out * dout) for the forward
    attn_fwd computes with the same arguments; out and lse are that forward's results. `workspace`
    (uint8, at least attn_bwd_workspace_bytes(...) bytes) is allocated when not given."""
    _check_input("q", q)
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, D]")
    B, T, H, D = q.shape
    _check_input("k", k)
    if k.dim() != 4 or k.shape[0] != B or k.shape[1] != T or k.shape[3] != D:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [B, T, H_kv, D] = [{B}, {T}, H_kv, {D}]")
    H_kv = k.shape[2]
    if H_kv < 1 or H % H_kv != 0:
        raise ValueError(f"H = {H} is not a multiple of H_kv = {H_kv}")
    _check_input("v", v, k.shape)
    _check_input("out", out, q.shape)
    _check_input("dout", dout, q.shape)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, T) or \
            lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 [B, H, T] tensor on q's device")
    nbytes = attn_bwd_workspace_bytes(B, H, H_kv, T, D)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or not workspace.is_contiguous() or workspace.numel() < nbytes:
        raise ValueError(f"workspace must be a contiguous uint8 tensor of at least {nbytes} bytes")

    def grad(t, name, shape):
        if t is None:
            return torch.empty(shape, dtype=torch.float32, device=q.device)
        if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must be a contiguous float32 tensor of shape {tuple(shape)}")
        return t

    dq = grad(dq, "dq", q.shape)
    dk = grad(dk, "dk", k.shape)
    dv = grad(dv, "dv", k.shape)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), workspace.numel(), B, H, H_kv,
                      T, D, int(window), int(bool(causal)), float(rope_base), float(eps),
                      ctypes.c_void_p(s.cuda_stream or None))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd_ve(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, ve: torch.Tensor, x_gate: torch.Tensor,
                w_gate: torch.Tensor, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
                eps: float = 1e-6, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """attn_fwd on a layer with value embeddings: v' = v + 2 sigmoid(x_gate[..., :32] @ w_gate.T) ve applied
    inside the kernel. ve like v ([B, T, H_kv, D] bf16); x_gate [B, T, C] bf16 with C >= 32 whose rows may be
    strided (a slice of x), last dimension contiguous; w_gate [H_kv, 32] bf16."""
    _check_input("q", q)
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, D]")
    B, T, H, D = q.shape
    _check_input("k", k)
    H_kv = k.shape[2]
    if k.dim() != 4 or tuple(k.shape) != (B, T, H_kv, D) or H % H_kv != 0:
        raise ValueError(f"k has shape {tuple(k.shape)}, expected [B, T, H_kv, D] with H a multiple of H_kv")
    _check_input("v", v, k.shape)
    _check_input("ve", ve, k.shape)
    if not isinstance(x_gate, torch.Tensor) or x_gate.device.type != "cuda" or x_gate.dtype != torch.bfloat16:
        raise ValueError("x_gate must be a bf16 CUDA tensor")
    if x_gate.dim() != 3 or tuple(x_gate.shape[:2]) != (B, T) or x_gate.shape[2] < 32 or x_gate.stride(2) != 1 \
            or x_gate.stride(0) != T * x_gate.stride(1):
        raise ValueError("x_gate must be [B, T, C >= 32] with contiguous rows of a common stride")
    _check_input("w_gate", w_gate, (H_kv, 32))
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_input("out", out, q.shape)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    nbytes = int(lib.attn_fwd_ve_workspace_bytes(B, H_kv, T))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    elif workspace.dtype != torch.uint8 or not workspace.is_contiguous() or workspace.numel() < nbytes:
        raise ValueError(f"workspace must be a contiguous uint8 tensor of at least {nbytes} bytes")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    rc = lib.attn_fwd_ve(q.data_ptr(), k.data_ptr(), v.data_ptr(), ve.data_ptr(), x_gate.data_ptr(),
                         x_gate.stride(1), w_gate.data_ptr(), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                         workspace.numel(), B, H, H_kv, T, D,
                         int(window), int(bool(causal)), float(rope_base), float(eps),
                         ctypes.c_void_p(s.cuda_stream or None))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_ve")
    return out, lse


def attn_fwd_ve_workspace_bytes(B: int, H_kv: int, T: int) -> int:
    return int(lib.attn_fwd_ve_workspace_bytes(B, H_kv, T))
