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

With round_qk=True the derivative is evaluated where the listing evaluates it: its autocast forward
rounds q^ and k^ to bf16 and saves the rounded tensors, and the cast passes the gradient through
unchanged. Scores, weights and the dq^ / dk^ products then use the rounded q^, k^ (the forward oracle's
rounding), while the norm and RoPE backward use the unrounded rotation and scale.

With return_tol=True the function also returns, per gradient element, a bound on how far an
implementation that rounds its MMA operands to bf16 may lie from this value: one that computes P and
dS = P (dP - delta) in fp32 and rounds each to bf16 (relative error at most u = 2^-8) for the
products dV = P^T dO, dk^ = dS^T q^ / sqrt(D) and dq^ = dS k^ / sqrt(D), and takes
delta_i = dO_i . out_i from the bf16 output (out rounded: |d delta_i| <= u sum_d |dO_id| |o_id|):
  |d dV_jd|  <= u sum_i p_ij |dO_id|
  |d dS_ij|  <= u |dS_ij| + p_ij |d delta_i|            (+ the fp32 rounding of the exponent, ~2^-22 p)
  |d dk^_jd| <= sum_i |d dS_ij| |q^_id| / sqrt(D),  |d dq^_id| <= sum_j |d dS_ij| |k^_jd| / sqrt(D)
and through the norm and RoPE backward, which are linear in dk^ / dq^ (dx = R^T (r dy - (r^3 / D)
(rx . dy) rx)), the bound of each element of dx is that map applied to the bounds with every term in
absolute value. The bound is returned multiplied by 2 (accumulation in fp32 and the fp32 evaluation of
the norm and rotation are far below it).

Pinned by tests/test_oracle_backward.py: the float64 forward here against the C forward oracle
(bit patterns in, without the bf16 rounding of q^, k^), central finite differences of that forward,
PyTorch autograd on a plain float64 implementation, and the zero-sum rows of the softmax Jacobian;
the rounded mode by autograd through a straight-through rounding of q^, k^, and the bound by
perturbing P and dS within it.
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


def _abs_prologue_back(tol: np.ndarray, rx: np.ndarray, r: np.ndarray, ang, eps: float) -> np.ndarray:
    """The norm + RoPE backward map with every coefficient in absolute value, applied to non-negative
    element bounds: an upper bound of |J dy| over all |dy| <= tol (J the map of _prologue_back)."""
    D = rx.shape[-1]
    if eps >= 0:
        t = r * tol + (r ** 3 / D) * np.sum(np.abs(rx) * tol, axis=-1, keepdims=True) * np.abs(rx)
    else:
        t = tol
    if ang is None:
        return t
    d = D // 2
    c, s = np.abs(np.cos(ang)), np.abs(np.sin(ang))
    t1, t2 = t[..., :d], t[..., d:]
    return np.concatenate([t1 * c + t2 * s, t1 * s + t2 * c], axis=-1)


def attn_bwd(q, k, v, dout, window: int = -1, causal: bool = True, rope_base: float = 10000.0,
             eps: float = 1e-6, round_qk: bool = False, return_tol: bool = False, out_used=None, lse_used=None):
    """Gradients (dq [B, T, H, D], dk, dv [B, T, Hkv, D]) of sum(out * dout) for the float64 forward.

    round_qk: evaluate at the bf16-rounded q^, k^ of the forward oracle (q, k must then be bf16
    tensors or uint16 bit patterns). return_tol (needs round_qk): also (tol_dq, tol_dk, tol_dv), the
    element bounds of the bf16-operand implementation described in the module docstring, for inputs
    out rounded to bf16 and lse rounded to fp32; or, when given, for the out ([B, T, H, D]) and lse
    ([B, H, T], natural log) the implementation was actually handed (a forward's own results): delta
    then moves by sum_d |dO_id| |out_used_id - out_id| and every weight of row i by the factor
    exp(|lse_used_i - lse_i|) - 1 (first order: the difference itself)."""
    assert round_qk or not return_tol, "the bounds describe the rounded evaluation"
    if round_qk:
        from . import qk_prologue

        qh_all, aq_all = qk_prologue(q, rope_base, eps, round_qk=True, return_amb=True)
        kh_all, ak_all = qk_prologue(k, rope_base, eps, round_qk=True, return_amb=True)
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    ang = _angles(T, D, rope_base) if rope_base > 0 else None
    ok = _allowed(T, window, causal)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    tq, tk, tv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    sc = 1.0 / np.sqrt(D)
    u = 2.0 ** -8      # bf16 rounding (8 significant bits), relative
    f = 2.0 ** -24     # fp32 rounding, relative
    fp32_map = (2 * D + 16) * f    # fp32 evaluation of the norm and rotation backward, relative
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            qh, rq, r_q = _prologue(q[b, :, h], ang, eps)
            kh, rk, r_k = _prologue(k[b, :, hk], ang, eps)
            if round_qk:
                qh, kh = qh_all[b, :, h], kh_all[b, :, hk]
            s = np.where(ok, qh @ kh.T * sc, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.where(ok, np.exp(s - m), 0.0)
            z = e.sum(axis=1, keepdims=True)
            p = e / z
            o = p @ v[b, :, hk]
            do = dout[b, :, h]
            dv[b, :, hk] += p.T @ do
            dp = do @ v[b, :, hk].T
            delta = np.sum(do * o, axis=1, keepdims=True)
            ds = p * (dp - delta)
            dqh = ds @ kh * sc
            dkh = ds.T @ qh * sc
            dq[b, :, h] = _prologue_back(dqh, rq, r_q, ang, eps)
            dk[b, :, hk] += _prologue_back(dkh, rk, r_k, ang, eps)
            if return_tol:
                aq, ak = aq_all[b, :, h], ak_all[b, :, hk]
                aqk, ak_ = np.abs(qh), np.abs(kh)
                lse = m + np.log(z)
                s0 = np.where(ok, s, 0.0)
                lse_move = 0.0 if lse_used is None else np.abs(_as_f64(lse_used)[b, h][:, None] - lse)
                # relative error of each weight P_ij = exp(s_ij - lse_i) before its bf16 rounding
                eta = ((aq @ ak_.T + aqk @ ak.T + aq @ ak.T) * sc      # other valid roundings of q^, k^
                       + D * f * (aqk @ ak_.T) * sc                     # fp32 accumulation of the score
                       + 4 * f * (1.0 + np.abs(s0) + np.abs(lse))       # lse in fp32, scaling, exp2
                       + lse_move)                                      # the lse handed in
                eta = np.where(ok, eta, 0.0)
                tv[b, :, hk] += ((u + eta + T * f) * p).T @ np.abs(do)
                d_dp = D * f * (np.abs(do) @ np.abs(v[b, :, hk]).T)
                if out_used is None:
                    d_delta = (u + D * f) * np.sum(np.abs(do) * np.abs(o), axis=1, keepdims=True)
                else:
                    d_delta = (np.sum(np.abs(do) * np.abs(_as_f64(out_used)[b, :, h] - o), axis=1, keepdims=True)
                               + D * f * np.sum(np.abs(do) * np.abs(o), axis=1, keepdims=True))
                d_ds = (u + 2 * f) * np.abs(ds) + eta * p * np.abs(dp - delta) + p * (d_dp + d_delta)
                d_ds = np.where(ok, d_ds, 0.0)
                t_dqh = (d_ds @ ak_ + np.abs(ds) @ ak + T * f * (np.abs(ds) @ ak_)) * sc
                t_dkh = (d_ds.T @ aqk + np.abs(ds).T @ aq + T * f * (np.abs(ds).T @ aqk)) * sc
                tq[b, :, h] = (_abs_prologue_back(t_dqh, rq, r_q, ang, eps)
                               + fp32_map * _abs_prologue_back(np.abs(dqh), rq, r_q, ang, eps))
                tk[b, :, hk] += (_abs_prologue_back(t_dkh, rk, r_k, ang, eps)
                                 + fp32_map * _abs_prologue_back(np.abs(dkh), rk, r_k, ang, eps))
    if return_tol:
        return dq, dk, dv, 2.0 * tq, 2.0 * tk, 2.0 * tv
    return dq, dk, dv
