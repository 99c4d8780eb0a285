"""The oracle: a plain float64 CPU reference of the attention forward pass.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package: only `tests/`,
`__graft_entry__.smoke()` and `bench.py`'s CPU-baseline / reference arm call it. It shares no
code with the CUDA path (see attn_oracle.c for the step-by-step definition and the passages
of the pages each step follows).

Every function takes q, k, v as bf16 tensors (CPU torch.bfloat16) or uint16 numpy arrays of
bf16 bit patterns: q in [B, T, H, D] layout, k and v in [B, T, Hkv, D] with H a multiple of Hkv
(grouped K/V heads: query head h uses K/V head h // (H // Hkv); Hkv = H is multi-head attention),
and returns float64 numpy arrays.

The prologue (RoPE, QK-norm) is evaluated in float64 in the listing's order and then rounded
to bf16. Where an exact value lies so close to a bf16 rounding midpoint that a single-precision
evaluation may round it the other way, both roundings are correct; `qk_prologue(...,
return_amb=True)` reports each element's ambiguity radius, and `attn_fwd` / `attn_rows` with
`return_slack=True` report how far those choices can move each output element and each LSE
(attn_oracle.c, steps 3 and 6). Everything after the rounding is float64.

Parity status: every function here is pinned: the forward and its helpers, the grouped K/V heads
and the value-embedding gate by `tests/test_oracle_pins.py` (worked example, closed forms,
invariants, library special cases, pure-Python brute force for T <= 8); the backward
(`attn_backward.py`) by `tests/test_oracle_backward.py` (finite differences, autograd); the Polar
Express orthogonalisation (`polar_express.py`) by `tests/test_oracle_polar.py` (SVD).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        ci, cd, cl = ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.oracle_attn_fwd.argtypes = [u16p, u16p, u16p, f64p, f64p, f64p, f64p, ci, ci, ci, ci, ci, ci, ci, cd,
                                        cd, ci, cd, ci]
        lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p, i32p, cl, f64p, f64p, f64p, f64p, ci, ci, ci, ci, ci,
                                         ci, ci, cd, cd, ci, cd, ci]
        lib.oracle_attn_probs.argtypes = [u16p, u16p, u16p, ci, ci, f64p, ci, ci, ci, ci, ci, ci, ci, cd, cd, ci]
        lib.oracle_qk_prologue.argtypes = [u16p, f64p, f64p, ci, ci, ci, ci, cd, cd, ci, cd, ci]
        lib.oracle_round_bf16.argtypes = [cd]
        lib.oracle_round_bf16.restype = cd
        lib.oracle_num_threads.restype = ci
        for f in (lib.oracle_attn_fwd, lib.oracle_attn_rows, lib.oracle_attn_probs, lib.oracle_qk_prologue):
            f.restype = ci
        _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 numpy array (no copy of values)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16, x.dtype
        return np.ascontiguousarray(x)
    import torch

    assert x.dtype == torch.bfloat16, x.dtype
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")


def num_threads() -> int:
    return _load().oracle_num_threads()


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned as float64."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).ravel()
    return np.array([lib.oracle_round_bf16(float(t)) for t in flat]).reshape(np.shape(x))


def qk_prologue(x, rope_base: float = 10000.0, eps: float = 1e-6, round_qk: bool = True,
                nthreads: int = 0, return_amb: bool = False, amb_scale: float = 1.0):
    """RoPE then RMSNorm of every [.., D] row of x ([B, T, H, D]), rounded to bf16; float64
    [B, T, H, D]. With return_amb, also the ambiguity radius of every element (attn_oracle.c,
    step 3; amb_scale multiplies the evaluation budget, 1 for the stated one)."""
    xb = _bits(x)
    B, T, H, D = xb.shape
    y = np.empty((B, T, H, D), dtype=np.float64)
    amb = np.empty((B, T, H, D), dtype=np.float64) if return_amb else None
    _check(_load().oracle_qk_prologue(_p(xb, ctypes.c_uint16), _p(y, ctypes.c_double),
                                      _p(amb, ctypes.c_double) if return_amb else None, B, T, H, D,
                                      float(rope_base), float(eps), int(round_qk), float(amb_scale),
                                      int(nthreads)))
    return (y, amb) if return_amb else y


def _kv_heads(qb, kb, vb) -> int:
    B, T, H, D = qb.shape
    Hkv = kb.shape[2]
    assert kb.shape == (B, T, Hkv, D) and vb.shape == kb.shape, "k, v must be [B, T, Hkv, D]"
    assert 1 <= Hkv <= H and H % Hkv == 0, "H must be a multiple of Hkv"
    return Hkv


def attn_fwd(q, k, v, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
             eps: float = 1e-6, round_qk: bool = True, nthreads: int = 0, return_slack: bool = False,
             amb_scale: float = 1.0):
    """Full forward. Returns (out float64 [B, T, H, D], lse float64 [B, H, T], natural log), and
    with return_slack also (out_slack [B, T, H, D], lse_slack [B, H, T]): how far the near-tie
    choices of q^, k^ can move each value (attn_oracle.c, step 6; amb_scale widens step 3's budget
    for tests)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, T, H, D = qb.shape
    Hkv = _kv_heads(qb, kb, vb)
    out = np.empty((B, T, H, D), dtype=np.float64)
    lse = np.empty((B, H, T), dtype=np.float64)
    os_ = np.empty((B, T, H, D), dtype=np.float64) if return_slack else None
    ls_ = np.empty((B, H, T), dtype=np.float64) if return_slack else None
    _check(_load().oracle_attn_fwd(_p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
                                   _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                   _p(os_, ctypes.c_double) if return_slack else None,
                                   _p(ls_, ctypes.c_double) if return_slack else None, B, H, Hkv, T, D,
                                   int(window), int(bool(causal)), float(rope_base), float(eps),
                                   int(round_qk), float(amb_scale), int(nthreads)))
    return (out, lse, os_, ls_) if return_slack else (out, lse)


def attn_rows(q, k, v, rows, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
              eps: float = 1e-6, round_qk: bool = True, nthreads: int = 0, return_slack: bool = False,
              amb_scale: float = 1.0):
    """Selected query rows only. rows: int array [n, 3] of (b, h, i).
    Returns (out float64 [n, D], lse float64 [n]), and with return_slack also
    (out_slack [n, D], lse_slack [n])."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, T, H, D = qb.shape
    Hkv = _kv_heads(qb, kb, vb)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    os_ = np.empty((n, D), dtype=np.float64) if return_slack else None
    ls_ = np.empty((n,), dtype=np.float64) if return_slack else None
    _check(_load().oracle_attn_rows(_p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
                                    _p(r, ctypes.c_int32), n, _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                                    _p(os_, ctypes.c_double) if return_slack else None,
                                    _p(ls_, ctypes.c_double) if return_slack else None,
                                    B, H, Hkv, T, D, int(window), int(bool(causal)), float(rope_base), float(eps),
                                    int(round_qk), float(amb_scale), int(nthreads)))
    return (out, lse, os_, ls_) if return_slack else (out, lse)


def attn_probs(q, k, v, b: int, h: int, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
               eps: float = 1e-6, round_qk: bool = True) -> np.ndarray:
    """The attention weight matrix p [T, T] (queries x keys) of head (b, h)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, T, H, D = qb.shape
    Hkv = _kv_heads(qb, kb, vb)
    p = np.empty((T, T), dtype=np.float64)
    _check(_load().oracle_attn_probs(_p(qb, ctypes.c_uint16), _p(kb, ctypes.c_uint16), _p(vb, ctypes.c_uint16),
                                     int(b), int(h), _p(p, ctypes.c_double), B, H, Hkv, T, D, int(window),
                                     int(bool(causal)), float(rope_base), float(eps), int(round_qk)))
    return p


def round_bf16_array(x) -> np.ndarray:
    """round_bf16 for whole float64 arrays: the nearest bf16 value (ties to even), by adding the
    rounding bias to the float64 bit pattern at the 8th significant bit. Values below the smallest
    normal bf16 (2^-126, none in this package's data but zero) go through round_bf16."""
    a = np.array(x, dtype=np.float64, copy=True)
    bits = a.view(np.uint64)
    keep = ~np.uint64((1 << 45) - 1)
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    out = ((bits + np.uint64((1 << 44) - 1) + lsb) & keep).view(np.float64)
    tiny = (np.abs(a) < 2.0 ** -126) & (a != 0.0)
    if tiny.any():
        out[tiny] = round_bf16(a[tiny])
    out[a == 0.0] = a[a == 0.0]
    return out


def _bf16_values(x) -> np.ndarray:
    b = _bits(x)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def value_gate(v, ve, x_gate, w_gate, return_amb: bool = False):
    """Value-embedding gate (habr "Autoresearch" deep dive, train.py listing, CausalSelfAttention.forward,
    "Value Residual (ResFormer)"): for every (b, t, K/V head h)
        gate = 2 * sigmoid(sum_c x_gate[b, t, c] * w_gate[h, c])      (c < 32 channels)
        v'   = v + gate * ve
    with each step rounded to bf16 as the listing's bf16 tensors are: the logit (the exact sum of the
    exact products, rounded once), the sigmoid (rounded once), x2 (exact), the product with ve
    (rounded), the sum with v (rounded). Everything else is float64.

    v, ve: [B, T, Hkv, D]; x_gate: [B, T, C]; w_gate: [Hkv, C] (bf16 tensors or uint16 bit patterns).
    Returns float64 [B, T, Hkv, D] holding bf16 values (the gated v the attention then reads).

    return_amb: also each element's ambiguity radius, the largest distance from v' to the v' of any
    evaluation whose logit and sigmoid are single-precision evaluations within these budgets: the
    logit accumulated over the 32 exact products in any order (each addition rounded: at most
    32 * 2^-24 * sum |x w| from the exact sum); the sigmoid 1 / (1 + exp(-logit)) with exp within 2 ulp
    and the addition and reciprocal correctly rounded (relative error at most 2^-21); the sum v + product
    either exact or first rounded to single precision. Each of those values is rounded to bf16 as above;
    the product gate * ve of two bf16 values is exact in single precision, so its rounding is unique."""
    vv, ee = _bf16_values(v), _bf16_values(ve)
    xx, ww = _bf16_values(x_gate), _bf16_values(w_gate)
    B, T, Hkv, D = vv.shape
    assert ee.shape == vv.shape and xx.shape[:2] == (B, T) and ww.shape == (Hkv, xx.shape[2])
    logit = np.empty((B, T, Hkv))
    mag = np.empty((B, T, Hkv))
    import math

    for b in range(B):
        for t in range(T):
            for h in range(Hkv):
                # products of two bf16 values are exact in float64; fsum adds them with one rounding
                terms = [float(a) * float(w) for a, w in zip(xx[b, t], ww[h])]
                logit[b, t, h] = math.fsum(terms)
                mag[b, t, h] = math.fsum(abs(z) for z in terms)

    def gated(lg):
        sig = round_bf16_array(1.0 / (1.0 + np.exp(-lg)))
        return sig

    lb = round_bf16_array(logit)
    sig = gated(lb)
    gate = 2.0 * sig
    prod = round_bf16_array(gate[..., None] * ee)
    out = round_bf16_array(vv + prod)
    if not return_amb:
        return out
    amb = np.zeros_like(out)
    budget = 32.0 * 2.0 ** -24 * mag
    for lg in (round_bf16_array(logit - budget), lb, round_bf16_array(logit + budget)):
        s_exact = 1.0 / (1.0 + np.exp(-lg))
        for sg in (round_bf16_array(s_exact * (1.0 - 2.0 ** -21)), round_bf16_array(s_exact),
                   round_bf16_array(s_exact * (1.0 + 2.0 ** -21))):
            pr = round_bf16_array((2.0 * sg)[..., None] * ee)
            s64 = vv + pr
            for cand in (round_bf16_array(s64), round_bf16_array(s64.astype(np.float32).astype(np.float64))):
                amb = np.maximum(amb, np.abs(cand - out))
    return out, amb


from .attn_backward import attn_bwd, attn_fwd_f64  # noqa: E402  (backward oracle, NEXT-1)

__all__ = ["attn_fwd", "attn_rows", "attn_probs", "qk_prologue", "round_bf16", "num_threads", "value_gate",
           "attn_bwd", "attn_fwd_f64"]
