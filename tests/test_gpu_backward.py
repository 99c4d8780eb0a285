"""GPU parity of the attention backward (attn_bwd through the C ABI) against the float64 backward oracle.

Both sides get the same inputs: q, k, v, dout in bf16 from the seeded generators, and the forward's
out and lse as the oracle computes them (out rounded to bf16, lse to fp32, which is what a forward
hands the backward). The oracle differentiates at the bf16-rounded q^, k^ (the listing's autocast
forward) and bounds, element by element, how far a backward that rounds P and dS to bf16 for its
products may lie from the exact value (oracle/attn_backward.py); every element must lie within
that bound. The bound also covers the near-tie roundings of q^, k^ (either neighbour is correct).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import attn_backward as ob
from sliding_window_attention_04_b300.inputs import make_qkv

pytestmark = pytest.mark.gpu

RATIO_LOG = []  # (case, max err / bound for dq, dk, dv)


@pytest.fixture(scope="module")
def attn():
    from sliding_window_attention_04_b300 import attn as a

    a.attn_init(0)
    return a


def make_inputs(B, T, H, Hkv, D, seed):
    q, _, _ = make_qkv(B, T, H, D, seed=seed)
    _, k, v = make_qkv(B, T, Hkv, D, seed=seed + 1)
    dout = make_qkv(B, T, H, D, seed=seed + 2)[2]
    return q, k, v, dout


def gpu_bwd(attn, q, k, v, dout, out_ref, lse_ref, window, causal, base, eps):
    out_b = torch.from_numpy(out_ref).to(torch.bfloat16).cuda()
    lse_f = torch.from_numpy(lse_ref).to(torch.float32).cuda()
    dq, dk, dv = attn.attn_bwd(q.cuda(), k.cuda(), v.cuda(), out_b, lse_f, dout.cuda(), window=window, causal=causal,
                               rope_base=base, eps=eps)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == 0
    return dq.cpu().double().numpy(), dk.cpu().double().numpy(), dv.cpu().double().numpy()


def compare(name, got, ref):
    ratios = []
    for what, g, (r, tol) in zip(("dq", "dk", "dv"), got, ref):
        err = np.abs(g - r)
        assert np.all(np.isfinite(g)), f"{name}: {what} has non-finite values"
        bad = err > tol
        assert not bad.any(), (f"{name}: {what} outside the bound at {np.argwhere(bad)[:5].tolist()}: "
                               f"err {err[bad][:5]} bound {tol[bad][:5]}")
        ratios.append(float((err / np.maximum(tol, 1e-300)).max()))
    RATIO_LOG.append((name, *ratios))


def oracle_bwd(q, k, v, dout, window, causal, base, eps):
    dq, dk, dv, tq, tk, tv = ob.attn_bwd(q, k, v, dout, window, causal, base, eps, round_qk=True, return_tol=True)
    return (dq, tq), (dk, tk), (dv, tv)


CASES = [  # (B, T, H, Hkv, D, window, causal, rope_base, eps)
    (1, 8, 2, 2, 32, 3, True, 10000.0, 1e-6),
    (1, 1, 2, 2, 64, -1, True, 10000.0, 1e-6),
    (2, 300, 2, 2, 64, 100, True, 10000.0, 1e-6),
    (1, 256, 2, 2, 32, -1, True, 10000.0, 1e-6),
    (1, 300, 4, 2, 64, 150, True, 10000.0, 1e-6),
    (1, 200, 2, 2, 128, 64, True, 10000.0, 1e-6),
    (1, 384, 2, 2, 64, 100, False, 10000.0, 1e-6),
    (1, 130, 2, 2, 64, -1, True, 0.0, -1.0),
    (1, 640, 2, 2, 64, 0, True, 10000.0, 1e-6),
    (1, 520, 4, 1, 128, 200, True, 500.0, 1e-6),
    # odd row counts (111 q rows, 37 k rows): ragged last groups of the staged prologue and finalize
    (1, 37, 3, 1, 32, 16, True, 10000.0, 1e-6),
    (3, 45, 3, 3, 64, 20, True, 10000.0, 1e-6),
]


@pytest.mark.parametrize("B,T,H,Hkv,D,window,causal,base,eps", CASES)
def test_backward_matches_oracle(attn, B, T, H, Hkv, D, window, causal, base, eps):
    q, k, v, dout = make_inputs(B, T, H, Hkv, D, 1000 + T + D)
    out_ref, lse_ref = oracle.attn_fwd(q, k, v, window=window, causal=causal, rope_base=base, eps=eps)
    got = gpu_bwd(attn, q, k, v, dout, out_ref, lse_ref, window, causal, base, eps)
    ref = oracle_bwd(q, k, v, dout, window, causal, base, eps)
    compare(f"B{B} T{T} H{H}/{Hkv} D{D} W{window} c{int(causal)}", got, ref)


def test_backward_workspace_reuse_and_gqa_sums(attn):
    """Two calls through one caller-owned workspace give identical dk, dv (deterministic) and dq within
    the bound; with H_kv = 1 the K/V gradients sum all query heads."""
    B, T, H, Hkv, D, W = 1, 384, 4, 1, 64, 128
    q, k, v, dout = make_inputs(B, T, H, Hkv, D, 77)
    out_ref, lse_ref = oracle.attn_fwd(q, k, v, window=W, causal=True)
    ws = torch.empty(attn.attn_bwd_workspace_bytes(B, H, Hkv, T, D), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)  # the workspace's contents on entry do not matter
    args = (q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(out_ref).to(torch.bfloat16).cuda(),
            torch.from_numpy(lse_ref).float().cuda(), dout.cuda())
    r1 = [t.clone() for t in attn.attn_bwd(*args, window=W, workspace=ws)]
    r2 = attn.attn_bwd(*args, window=W, workspace=ws)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == 0
    assert torch.equal(r1[1], r2[1]) and torch.equal(r1[2], r2[2])
    ref = oracle_bwd(q, k, v, dout, W, True, 10000.0, 1e-6)
    for got in (r1, r2):
        compare("workspace reuse", tuple(t.cpu().double().numpy() for t in got), ref)


def test_backward_through_the_forward_kernel(attn):
    """The user's path: out and lse from attn_fwd, then attn_bwd. The oracle's bounds are taken for the
    out and lse the backward was handed (their distance from the exact ones moves delta and P)."""
    B, T, H, Hkv, D, W = 2, 512, 2, 2, 64, 256
    q, k, v, dout = make_inputs(B, T, H, Hkv, D, 4242)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    out, lse = attn.attn_fwd(qc, kc, vc, window=W, causal=True)
    dq, dk, dv = attn.attn_bwd(qc, kc, vc, out, lse, dout.cuda(), window=W)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == 0
    out_used = out.cpu().double().numpy()
    lse_used = lse.cpu().double().numpy()
    r = ob.attn_bwd(q, k, v, dout, W, True, 10000.0, 1e-6, round_qk=True, return_tol=True, out_used=out_used,
                    lse_used=lse_used)
    compare("through attn_fwd", (dq.cpu().double().numpy(), dk.cpu().double().numpy(), dv.cpu().double().numpy()),
            ((r[0], r[3]), (r[1], r[4]), (r[2], r[5])))


@pytest.mark.parametrize("heads", [[(0, 0), (5, 7), (31, 11)]])
def test_backward_andrea120m_layer_sampled_heads(attn, heads):
    """The ANDREA-120M shape (B=32, H=12, T=1024, D=64), one S layer (W=512) at full size: the oracle's
    forward for every head feeds the GPU backward; three (batch row, head) pairs are checked whole
    against the backward oracle."""
    B, T, H, D, W = 32, 1024, 12, 64, 512
    q, k, v, dout = make_inputs(B, T, H, H, D, 2024)
    out_ref, lse_ref = oracle.attn_fwd(q, k, v, window=W, causal=True)
    got = gpu_bwd(attn, q, k, v, dout, out_ref, lse_ref, W, True, 10000.0, 1e-6)
    for b, h in heads:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ref = oracle_bwd(q[sl].contiguous(), k[sl].contiguous(), v[sl].contiguous(), dout[sl].contiguous(), W, True,
                         10000.0, 1e-6)
        compare(f"120M b{b} h{h}", tuple(g[sl] for g in got), ref)


def test_backward_rejects_unsupported(attn):
    q, k, v, dout = make_inputs(1, 64, 2, 2, 48, 5)
    with pytest.raises(attn.AttnError):
        attn.attn_bwd(q.cuda(), k.cuda(), v.cuda(), q.cuda(), torch.zeros(1, 2, 64, device="cuda"), dout.cuda())
