"""Oracle for the attention backward pass: float64 gradients of the forward with respect to q, k, v.

TEST INFRASTRUCTURE ONLY, like the rest of this package: nothing in the product path imports it,
and it shares no code with the CUDA path.

The pages train the model (habr "Autoresearch" deep dive, train.py listing: the training step calls
loss.backward() through CausalSelfAttention.forward, i.e. apply_rotary_emb, norm() and the attention
call). The backward of the attention forward is therefore the derivative of the function the forward
oracle defines (attn_oracle.c, steps 1-5). It is taken here in float64 without the bf16 rounding of
q^ and k^: casts pass gradients through unchanged in autograd, so the listing's backward is this
derivative evaluated at its rounded saved tensors.

Forward, per batch row b and query head h (K/V head hk = h // (H // Hkv)):
    rq = RoPE(q)  (pairs (i, i + D/2) rotated by the angle t * base^(-2i/D); identity if base <= 0)
    q^ = rq / sqrt(mean(rq^2) + eps)          (no norm if eps < 0); the same for k
    s  = q^ k^T / sqrt(D) on the allowed keys J(i), p = softmax(s) row by row, out = p v
Backward, given dout = dL/dout:
    dv  = p^T dout                             (summed over the query heads sharing the K/V head)
    dp  = dout v^T
    ds  = p * (dp - rowsum(dout * out))        (the softmax Jacobian; zero outside J(i))
    dq^ = ds k^ / sqrt(D),  dk^ = ds^T q^ / sqrt(D)
    norm y = x r, r = (mean(x^2) + eps)^(-1/2):  dx = r dy - (r^3 / D) (x . dy) x
    RoPE rotates each pair by +angle, so its transpose rotates by -angle.

Pinned by tests/test_oracle_backward.py: the float64 forward here against the C forward oracle
(bit patterns in, without the bf16 rounding of q^, k^), central finite differences of that forward,
PyTorch autograd on a plain float64 implementation, and the zero-sum rows of the softmax Jacobian.
"""
from __future__ import annotations

import numpy as np


def _angles(T: int, D: int, base: float) -> np.ndarray:
    i = np.arange(D // 2, dtype=np.float64)
    return np.arange(T, dtype=np.float64)[:, None] * np.power(float(base), -2.0 * i / D)[None, :]  # [T, D/2]


def _rotate(x: np.ndarray, ang: np.ndarray, sign: float) -> np.ndarray:
    """Rotate the pairs (x[..., i], x[..., i + D/2]) of x [T, D] by sign * angle [T, D/2]."""
    d = x.shape[-1] // 2
    c, s = np.cos(ang), sign * np.sin(ang)
    x1, x2 = x[..., :d], x[..., d:]
    return np.concatenate([x1 * c + x2 * s, -x1 * s + x2 * c], axis=-1)


def _allowed(T: int, window: int, causal: bool) -> np.ndarray:
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    ok = np.ones((T, T), dtype=bool)
    if causal:
        ok &= j <= i
    if window >= 0:
        ok &= j >= i - window
        if not causal:
            ok &= j <= i + window
    return ok


def _prologue(x: np.ndarray, ang, eps: float):
    """x [T, D] -> (rotated, normalised x, rotated x, r per row)."""
    rx = _rotate(x, ang, +1.0) if ang is not None else x
    if eps >= 0:
        r = 1.0 / np.sqrt(np.mean(rx * rx, axis=-1, keepdims=True) + eps)
    else:
        r = np.ones((x.shape[0], 1))
    return rx * r, rx, r


def _prologue_back(dy: np.ndarray, rx: np.ndarray, r: np.ndarray, ang, eps: float) -> np.ndarray:
    D = rx.shape[-1]
    if eps >= 0:
        drx = r * dy - (r ** 3 / D) * np.sum(rx * dy, axis=-1, keepdims=True) * rx
    else:
        drx = dy
    return _rotate(drx, ang, -1.0) if ang is not None else drx


def _as_f64(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return x.astype(np.float64)
    return x.detach().cpu().to(dtype=__import__("torch").float64).numpy()


def attn_fwd_f64(q, k, v, window: int = -1, causal: bool = True, rope_base: float = 10000.0, eps: float = 1e-6):
    """The forward in float64 on real-valued inputs (q [B, T, H, D]; k, v [B, T, Hkv, D]), without any
    bf16 rounding. Returns (out [B, T, H, D], lse [B, H, T])."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    ang = _angles(T, D, rope_base) if rope_base > 0 else None
    ok = _allowed(T, window, causal)
    out = np.zeros((B, T, H, D))
    lse = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            qh, _, _ = _prologue(q[b, :, h], ang, eps)
            kh, _, _ = _prologue(k[b, :, hk], ang, eps)
            s = np.where(ok, qh @ kh.T / np.sqrt(D), -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.where(ok, np.exp(s - m), 0.0)
            z = e.sum(axis=1, keepdims=True)
            out[b, :, h] = (e / z) @ v[b, :, hk]
            lse[b, h] = (m + np.log(z))[:, 0]
    return out, lse


def attn_bwd(q, k, v, dout, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
             eps: float = 1e-6):
    """Gradients (dq [B, T, H, D], dk, dv [B, T, Hkv, D]) of sum(out * dout) for the float64 forward."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    ang = _angles(T, D, rope_base) if rope_base > 0 else None
    ok = _allowed(T, window, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    sc = 1.0 / np.sqrt(D)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            qh, rq, r_q = _prologue(q[b, :, h], ang, eps)
            kh, rk, r_k = _prologue(k[b, :, hk], ang, eps)
            s = np.where(ok, qh @ kh.T * sc, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.where(ok, np.exp(s - m), 0.0)
            p = e / e.sum(axis=1, keepdims=True)
            o = p @ v[b, :, hk]
            do = dout[b, :, h]
            dv[b, :, hk] += p.T @ do
            dp = do @ v[b, :, hk].T
            ds = p * (dp - np.sum(do * o, axis=1, keepdims=True))
            dqh = ds @ kh * sc
            dkh = ds.T @ qh * sc
            dq[b, :, h] = _prologue_back(dqh, rq, r_q, ang, eps)
            dk[b, :, hk] += _prologue_back(dkh, rk, r_k, ang, eps)
    return dq, dk, dv
