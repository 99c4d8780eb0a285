"""GPU parity of the value-embedding gate fused into the forward (attn_fwd_ve) against the oracle.

The oracle gates v (oracle.value_gate: every step rounded to bf16 as the listing's bf16 tensors are) and
runs its float64 forward on the gated values. Where a gate step's exact value lies within an fp32
evaluation's error of a bf16 midpoint either rounding is correct; the oracle reports each gated element's
ambiguity radius, and its effect on an output element, sum_j p_ij * radius_jd, widens that element's
tolerance (as the q^/k^ near-tie slack does).

The gated values reach |v'| ~ 9, twice the range of the plain inputs, and the forward's own error grows with
|v|: P is rounded to bf16 for the P.V product (at most half a bf16 step, 2^-9 relative, per weight) and the
output to bf16, so |out_gpu - out| <= 2^-9 (sum_j p_ij |v_jd| + |out_id|) to first order. Where twice that
bound exceeds the 2e-2 used for the plain inputs, it is the tolerance.

Where the oracle finds no near-tie at all, the gated kernel must equal the plain kernel run on the oracle's
gated values bit for bit: the gate inside the kernel then produced exactly the oracle's v'.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import OUT_ATOL, LSE_RTOL
from sliding_window_attention_04_b300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    from sliding_window_attention_04_b300 import attn as a

    a.attn_init(0)
    return a


def gate_inputs(B, T, H, Hkv, D, C, seed):
    q, _, _ = make_qkv(B, T, H, D, seed=seed)
    _, k, v = make_qkv(B, T, Hkv, D, seed=seed + 1)
    ve = make_qkv(B, T, Hkv, D, seed=seed + 2)[2]
    g = torch.Generator().manual_seed(seed + 3)
    x = torch.randn(B, T, C, generator=g).to(torch.bfloat16)
    w = (torch.randn(Hkv, 32, generator=g) * 0.3).to(torch.bfloat16)
    return q, k, v, ve, x, w


def check(attn, B, T, H, Hkv, D, C, window, causal, base, eps, heads=None, seed=0):
    q, k, v, ve, x, w = gate_inputs(B, T, H, Hkv, D, C, 7000 + T + D + seed)
    out, lse = attn.attn_fwd_ve(q.cuda(), k.cuda(), v.cuda(), ve.cuda(), x.cuda(), w.cuda(), window=window,
                                causal=causal, rope_base=base, eps=eps)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == 0
    vg, amb = oracle.value_gate(v, ve, x[..., :32].contiguous(), w, return_amb=True)
    vg_bf = torch.from_numpy(vg.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(vg_bf.to(torch.float64), torch.from_numpy(vg))  # exact bf16 values
    ref, lref, os_, ls_ = oracle.attn_fwd(q, k, vg_bf, window=window, causal=causal, rope_base=base, eps=eps,
                                          return_slack=True)
    got, lgot = out.cpu().double().numpy(), lse.cpu().double().numpy()
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    worst = 0.0
    for b, h in heads:
        hk = h // (H // Hkv)
        p = oracle.attn_probs(q, k, vg_bf, b, h, window=window, causal=causal, rope_base=base, eps=eps)
        vslack = p @ amb[b, :, hk, :]
        err = np.abs(got[b, :, h] - ref[b, :, h])
        fwd_bound = 2.0 * 2.0 ** -9 * (p @ np.abs(vg[b, :, hk, :]) + np.abs(ref[b, :, h]))
        tol = np.maximum(OUT_ATOL, fwd_bound) + os_[b, :, h] + vslack
        assert np.all(err <= tol), (b, h, float((err - tol).max()))
        lerr = np.abs(lgot[b, h] - lref[b, h])
        assert np.all(lerr <= LSE_RTOL * np.maximum(1.0, np.abs(lref[b, h])) + ls_[b, h]), (b, h)
        worst = max(worst, float(err.max()))
    # the gate changes the result: the plain forward on the ungated v differs
    plain, _ = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), window=window, causal=causal, rope_base=base, eps=eps)
    assert float((plain - out).abs().max()) > 10 * OUT_ATOL
    # no near-tie anywhere: the kernel's gated values are the oracle's, so the plain kernel on them agrees bitwise
    if not amb.any():
        same, lsame = attn.attn_fwd(q.cuda(), k.cuda(), vg_bf.cuda(), window=window, causal=causal, rope_base=base,
                                    eps=eps)
        torch.cuda.synchronize()
        assert torch.equal(same, out) and torch.equal(lsame, lse)
    return worst, float(amb.max())


@pytest.mark.parametrize("B,T,H,Hkv,D,C,window,causal,base,eps", [
    (1, 200, 2, 2, 64, 32, 100, True, 10000.0, 1e-6),
    (2, 300, 4, 2, 64, 64, 150, True, 10000.0, 1e-6),     # x rows strided (C = 64), grouped K/V heads
    (1, 256, 2, 2, 32, 32, -1, True, 10000.0, 1e-6),
    (1, 200, 2, 1, 128, 40, 64, True, 10000.0, 1e-6),     # D = 128, stride 40
    (1, 130, 2, 2, 64, 32, -1, True, 0.0, -1.0),          # raw mode (running-max softmax)
    (1, 384, 2, 2, 64, 32, 100, False, 10000.0, 1e-6),    # non-causal window
])
def test_value_gate_forward_matches_oracle(attn, B, T, H, Hkv, D, C, window, causal, base, eps):
    check(attn, B, T, H, Hkv, D, C, window, causal, base, eps)


def test_value_gate_forward_120m_layer_sampled_heads(attn):
    """A 120M-shaped S layer (B = 8 of 32 batch rows, H = 12, T = 1024, D = 64, W = 512), x rows from a 768-wide
    activation (stride 768); three (batch row, head) pairs compared whole."""
    check(attn, 8, 1024, 12, 12, 64, 768, 512, True, 10000.0, 1e-6, heads=[(0, 0), (3, 5), (7, 11)])


def test_value_gate_forward_whole_head_tickets(attn):
    """B = 16, H = 12, T = 1024, W = 512: 192 heads, so the kernel runs the first 44 as whole-head tickets
    (every query block of the head on one CTA, key tiles shared across its blocks) and the rest as pairs;
    the first and the last whole-head ticket's heads and the last head (a pair) are compared whole."""
    check(attn, 16, 1024, 12, 12, 64, 768, 512, True, 10000.0, 1e-6, heads=[(0, 0), (3, 7), (15, 11)], seed=5)


def test_value_gate_leaves_inputs_and_plain_path_unchanged(attn):
    q, k, v, ve, x, w = gate_inputs(1, 256, 2, 2, 64, 32, 99)
    qc, kc, vc, vec = q.cuda(), k.cuda(), v.cuda(), ve.cuda()
    v0 = vc.clone()
    a, la = attn.attn_fwd(qc, kc, vc, window=128)
    attn.attn_fwd_ve(qc, kc, vc, vec, x.cuda(), w.cuda(), window=128)
    b, lb = attn.attn_fwd(qc, kc, vc, window=128)
    torch.cuda.synchronize()
    assert torch.equal(vc, v0)                       # v is read, never written
    assert torch.equal(a, b) and torch.equal(la, lb)  # the ungated path after a gated call is unchanged
