"""Pins of the backward oracle (oracle/attn_backward.py), CPU only.

- its float64 forward equals the C forward oracle on the same bf16 inputs (without the bf16 rounding
  of q^ and k^), so it inherits that oracle's pins;
- the analytic gradients equal central finite differences of that forward;
- they equal PyTorch autograd on a plain float64 implementation of the same forward;
- every row of the softmax Jacobian sums to zero: shifting all scores of a row leaves the output,
  so the gradient with respect to q is zero when every key is the same vector (no RoPE, no norm).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import attn_backward as ob
from sliding_window_attention_04_b300.inputs import make_qkv

CASES = [  # (B, T, H, Hkv, D, window, causal, rope_base, eps)
    (1, 6, 2, 2, 8, 3, True, 10000.0, 1e-6),
    (2, 9, 2, 1, 8, -1, True, 500.0, 0.1),
    (1, 7, 3, 3, 4, 2, False, 10000.0, 1e-6),
    (1, 5, 2, 2, 8, -1, True, 0.0, -1.0),
]


def _inputs(B, T, H, Hkv, D, seed):
    q, _, _ = make_qkv(B, T, H, D, seed=seed)
    _, k, v = make_qkv(B, T, Hkv, D, seed=seed + 1)
    return q, k, v


@pytest.mark.parametrize("B,T,H,Hkv,D,window,causal,base,eps", CASES)
def test_f64_forward_matches_c_oracle(B, T, H, Hkv, D, window, causal, base, eps):
    q, k, v = _inputs(B, T, H, Hkv, D, 300 + T)
    out, lse = ob.attn_fwd_f64(q, k, v, window, causal, base, eps)
    ref, lref = oracle.attn_fwd(q, k, v, window=window, causal=causal, rope_base=base, eps=eps, round_qk=False)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,T,H,Hkv,D,window,causal,base,eps", CASES)
def test_gradients_match_finite_differences(B, T, H, Hkv, D, window, causal, base, eps):
    q, k, v = (ob._as_f64(t) for t in _inputs(B, T, H, Hkv, D, 400 + T))
    rng = np.random.default_rng(T)
    dout = rng.standard_normal(q.shape)
    dq, dk, dv = ob.attn_bwd(q, k, v, dout, window, causal, base, eps)

    def loss(qq, kk, vv):
        return float(np.sum(ob.attn_fwd_f64(qq, kk, vv, window, causal, base, eps)[0] * dout))

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def _torch_forward(q, k, v, window, causal, base, eps):
    """A plain float64 PyTorch forward with the listing's RoPE formula and RMSNorm, for autograd."""
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    d = D // 2

    def rope(x):
        if base <= 0:
            return x
        i = torch.arange(d, dtype=torch.float64)
        ang = torch.arange(T, dtype=torch.float64)[:, None] * torch.pow(torch.tensor(float(base), dtype=torch.float64),
                                                                      -2.0 * i / D)[None, :]
        c, s = torch.cos(ang)[None, :, None, :], torch.sin(ang)[None, :, None, :]
        x1, x2 = x[..., :d], x[..., d:]
        return torch.cat([x1 * c + x2 * s, x1 * (-s) + x2 * c], 3)

    def norm(x):
        return x if eps < 0 else x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps)

    qh, kh = norm(rope(q)), norm(rope(k))
    kh = kh.repeat_interleave(H // Hkv, dim=2)
    vv = v.repeat_interleave(H // Hkv, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", qh, kh) / D ** 0.5
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    ok = torch.ones(T, T, dtype=torch.bool)
    if causal:
        ok &= j <= i
    if window >= 0:
        ok &= j >= i - window
        if not causal:
            ok &= j <= i + window
    p = torch.softmax(s.masked_fill(~ok, float("-inf")), dim=-1)
    return torch.einsum("bhij,bjhd->bihd", p, vv)


@pytest.mark.parametrize("B,T,H,Hkv,D,window,causal,base,eps", CASES)
def test_gradients_match_torch_autograd(B, T, H, Hkv, D, window, causal, base, eps):
    q, k, v = (t.to(torch.float64) for t in _inputs(B, T, H, Hkv, D, 500 + T))
    dout = torch.randn(q.shape, dtype=torch.float64, generator=torch.Generator().manual_seed(T))
    qt, kt, vt = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = _torch_forward(qt, kt, vt, window, causal, base, eps)
    np.testing.assert_allclose(out.detach().numpy(), ob.attn_fwd_f64(q, k, v, window, causal, base, eps)[0],
                               rtol=0, atol=1e-12)
    (out * dout).sum().backward()
    dq, dk, dv = ob.attn_bwd(q, k, v, dout, window, causal, base, eps)
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-11)


def test_dq_vanishes_when_all_keys_are_equal():
    """Raw mode, every key the same vector: all scores of a row are equal and stay equal when q moves,
    so the output does not depend on q (the softmax Jacobian rows sum to zero)."""
    q, _, v = _inputs(1, 8, 2, 2, 8, 77)
    k = torch.ones_like(q)
    dout = np.random.default_rng(1).standard_normal(q.shape)
    dq, _, _ = ob.attn_bwd(q, k, v, dout, -1, True, 0.0, -1.0)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)


ROUNDED_CASES = [  # (B, T, H, Hkv, D, window, causal, rope_base, eps)
    (1, 7, 2, 2, 8, 3, True, 10000.0, 1e-6),
    (1, 9, 4, 2, 16, -1, True, 500.0, 1e-6),
    (2, 6, 2, 1, 8, 2, False, 0.0, -1.0),
]


def _st_round(x, rounded):
    """Straight-through rounding: the value of `rounded`, the gradient of x (a bf16 cast under autograd)."""
    return x + (rounded - x).detach()


@pytest.mark.parametrize("B,T,H,Hkv,D,window,causal,base,eps", ROUNDED_CASES)
def test_rounded_mode_matches_straight_through_autograd(B, T, H, Hkv, D, window, causal, base, eps):
    """round_qk=True: the derivative of the forward whose q^, k^ are rounded to bf16 by a cast that passes
    gradients through unchanged, as autocast does."""
    q, k, v = _inputs(B, T, H, Hkv, D, 700 + T)
    qr = torch.from_numpy(oracle.qk_prologue(q, base, eps, round_qk=True))
    kr = torch.from_numpy(oracle.qk_prologue(k, base, eps, round_qk=True))
    dout = torch.randn(q.shape, dtype=torch.float64, generator=torch.Generator().manual_seed(T))
    qt, kt, vt = (t.to(torch.float64).requires_grad_(True) for t in (q, k, v))
    d = D // 2

    def prologue(x, rounded):
        if base > 0:
            i = torch.arange(d, dtype=torch.float64)
            ang = torch.arange(T, dtype=torch.float64)[:, None] * (float(base) ** (-2.0 * i / D))[None, :]
            c, s = torch.cos(ang)[None, :, None, :], torch.sin(ang)[None, :, None, :]
            x = torch.cat([x[..., :d] * c + x[..., d:] * s, -x[..., :d] * s + x[..., d:] * c], 3)
        if eps >= 0:
            x = x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps)
        return _st_round(x, rounded)

    qh = prologue(qt, qr)
    kh = prologue(kt, kr).repeat_interleave(H // Hkv, dim=2)
    vv = vt.repeat_interleave(H // Hkv, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", qh, kh) / D ** 0.5
    ok = torch.from_numpy(ob._allowed(T, window, causal))
    out = torch.einsum("bhij,bjhd->bihd", torch.softmax(s.masked_fill(~ok, float("-inf")), -1), vv)
    (out * dout).sum().backward()
    dq, dk, dv = ob.attn_bwd(q, k, v, dout, window, causal, base, eps, round_qk=True)
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-11)
    # the rounding moved the gradient (the mode is not a no-op) unless q, k pass the prologue unchanged
    dq0 = ob.attn_bwd(q, k, v, dout, window, causal, base, eps)[0]
    assert (np.abs(dq0 - dq).max() > 1e-6) == (eps >= 0)


@pytest.mark.parametrize("base,eps", [(10000.0, 1e-6), (0.0, 1e-6), (500.0, -1.0), (0.0, -1.0)])
def test_abs_backward_map_bounds_the_jacobian(base, eps):
    """_abs_prologue_back(t) >= |J| t for the linear map J of the norm + RoPE backward, with J read column by
    column off _prologue_back; without norm and RoPE J is the identity and the bound is exact."""
    T, D = 5, 8
    rng = np.random.default_rng(11)
    x = rng.standard_normal((T, D))
    ang = ob._angles(T, D, base) if base > 0 else None
    _, rx, r = ob._prologue(x, ang, eps)
    for _ in range(5):
        t = rng.random((T, D))
        absJt = np.zeros((T, D))
        for e in range(D):
            unit = np.zeros((T, D))
            unit[:, e] = 1.0
            absJt += np.abs(ob._prologue_back(unit, rx, r, ang, eps)) * t[:, e:e + 1]
        bound = ob._abs_prologue_back(t, rx, r, ang, eps)
        assert np.all(bound >= absJt * (1 - 1e-12))
        if base <= 0 and eps < 0:
            np.testing.assert_allclose(bound, absJt, rtol=1e-15)


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _emulated_kernel_grads(q, k, v, dout, window, causal, base, eps, sign_p=None, sign_ds=None, out_lse=None):
    """A bf16-operand backward in float32 numpy: P = exp(s - lse) from the fp32 lse, rounded to bf16 for
    dV; dS = P (dP - delta) with delta from the bf16 output, rounded to bf16 for dq^, dk^; the norm and
    RoPE backward in float32. sign_p / sign_ds (per b, h: [T, T] arrays of +-1) push P and dS by a full
    rounding unit in a chosen direction instead of rounding to nearest."""
    qh_all = oracle.qk_prologue(q, base, eps, round_qk=True)
    kh_all = oracle.qk_prologue(k, base, eps, round_qk=True)
    out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal, rope_base=base, eps=eps)
    if out_lse is not None:
        out, lse = out_lse
    qf, kf, vf, dof = (ob._as_f64(t) for t in (q, k, v, dout))
    B, T, H, D = qf.shape
    Hkv = kf.shape[2]
    ang = ob._angles(T, D, base) if base > 0 else None
    ok = ob._allowed(T, window, causal)
    f32 = np.float32
    dq, dk, dv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            qh, kh = qh_all[b, :, h].astype(f32), kh_all[b, :, hk].astype(f32)
            s = (qh @ kh.T) * f32(1 / np.sqrt(D))
            p = np.where(ok, np.exp(s - lse[b, h].astype(f32)[:, None]), f32(0)).astype(f32)
            do = dof[b, :, h].astype(f32)
            o = _bf16(out[b, :, h]).astype(f32)
            dp = do @ vf[b, :, hk].astype(f32).T
            ds = (p * (dp - np.sum(do * o, axis=1, keepdims=True))).astype(f32)
            pb = _bf16(p) if sign_p is None else p * (1 + 2.0 ** -8 * sign_p[b, h])
            dsb = _bf16(ds) if sign_ds is None else ds * (1 + 2.0 ** -8 * sign_ds[b, h])
            dv[b, :, hk] += (pb.astype(f32).T @ do)
            dqh = (dsb.astype(f32) @ kh) * f32(1 / np.sqrt(D))
            dkh = (dsb.astype(f32).T @ qh) * f32(1 / np.sqrt(D))
            _, rq, r_q = ob._prologue(qf[b, :, h], ang, eps)
            _, rk, r_k = ob._prologue(kf[b, :, hk], ang, eps)
            dq[b, :, h] = ob._prologue_back(dqh, rq.astype(f32), r_q.astype(f32), ang, eps)
            dk[b, :, hk] += ob._prologue_back(dkh, rk.astype(f32), r_k.astype(f32), ang, eps)
    return dq, dk, dv


@pytest.mark.parametrize("B,T,H,Hkv,D,window,causal,base,eps", ROUNDED_CASES)
def test_tolerance_covers_a_bf16_operand_backward(B, T, H, Hkv, D, window, causal, base, eps):
    """The element bounds hold (without their factor-2 margin) for an emulated bf16-operand backward,
    rounding to nearest and pushed by whole rounding units in random directions; and the dv bound is
    attained, to its first-order terms, by the pushes aligned with dout."""
    q, k, v = _inputs(B, T, H, Hkv, D, 900 + T)
    rng = np.random.default_rng(T + D)
    dout = torch.from_numpy(rng.standard_normal(q.shape)).to(torch.bfloat16)
    dq, dk, dv, tq, tk, tv = ob.attn_bwd(q, k, v, dout, window, causal, base, eps, round_qk=True,
                                         return_tol=True)
    runs = [_emulated_kernel_grads(q, k, v, dout, window, causal, base, eps)]
    for _ in range(3):
        sp = rng.choice([-1.0, 1.0], size=(B, H, T, T))
        sd = rng.choice([-1.0, 1.0], size=(B, H, T, T))
        runs.append(_emulated_kernel_grads(q, k, v, dout, window, causal, base, eps, sp, sd))
    for gq, gk, gv in runs:
        assert np.all(np.abs(gq - dq) <= tq / 2), np.max(np.abs(gq - dq) / tq)
        assert np.all(np.abs(gk - dk) <= tk / 2), np.max(np.abs(gk - dk) / tk)
        assert np.all(np.abs(gv - dv) <= tv / 2), np.max(np.abs(gv - dv) / tv)
    # pushes of P aligned with dout[..., d0] move dv[..., d0] by u sum_i p_ij |dout_id0| (and H / Hkv heads add)
    d0 = 1
    sp = np.sign(ob._as_f64(dout))[:, :, :, d0].transpose(0, 2, 1)[:, :, :, None] * np.ones((1, 1, 1, T))
    _, _, gv = _emulated_kernel_grads(q, k, v, dout, window, causal, base, eps, sp, None)
    moved = np.abs(gv - dv)[..., d0]
    assert np.all(moved <= tv[..., d0] / 2)
    assert np.max(moved / np.maximum(tv[..., d0] / 2, 1e-30)) > 0.6


def test_tolerance_follows_the_out_and_lse_handed_in():
    """With out_used / lse_used (a forward's own results, off the exact ones), the bounds hold for the
    emulated backward fed with them, and they exceed the plain bounds by the move those inputs cause."""
    B, T, H, Hkv, D, window, causal, base, eps = 1, 9, 2, 2, 8, 4, True, 10000.0, 1e-6
    q, k, v = _inputs(B, T, H, Hkv, D, 31)
    rng = np.random.default_rng(5)
    dout = torch.from_numpy(rng.standard_normal(q.shape)).to(torch.bfloat16)
    out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal, rope_base=base, eps=eps)
    out_used = _bf16(out + 0.01 * rng.standard_normal(out.shape))
    lse_used = (lse + 1e-4 * rng.choice([-1.0, 1.0], size=lse.shape)).astype(np.float32).astype(np.float64)
    dq, dk, dv, tq, tk, tv = ob.attn_bwd(q, k, v, dout, window, causal, base, eps, round_qk=True, return_tol=True,
                                         out_used=out_used, lse_used=lse_used)
    _, _, _, tq0, tk0, tv0 = ob.attn_bwd(q, k, v, dout, window, causal, base, eps, round_qk=True, return_tol=True)
    assert np.all(tq > tq0) and np.all(tk > tk0) and np.all(tv > tv0)
    gq, gk, gv = _emulated_kernel_grads(q, k, v, dout, window, causal, base, eps, out_lse=(out_used, lse_used))
    assert np.all(np.abs(gq - dq) <= tq / 2), np.max(np.abs(gq - dq) / tq)
    assert np.all(np.abs(gk - dk) <= tk / 2), np.max(np.abs(gk - dk) / tk)
    assert np.all(np.abs(gv - dv) <= tv / 2), np.max(np.abs(gv - dv) / tv)
    # the plain bounds do not cover this input: the pin sees the move
    assert (np.abs(gq - dq) > tq0 / 2).any() or (np.abs(gk - dk) > tk0 / 2).any()
