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
