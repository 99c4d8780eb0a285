"""Pins of the float64 oracle against what the pages and the mathematics fix (CPU only).

Each test would fail for a plausible mistake somewhere in the oracle: a dropped eps, a wrong
RoPE sign or pairing, an off-by-one in the window, a transposed operand, a wrong scale.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import brute
from sliding_window_attention_04_b300.configs import n_allowed_keys, n_unmasked
from sliding_window_attention_04_b300.inputs import make_qkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------------------------
# Worked example ("geometry_of_andrea", "Lendo uma Projeção")


def test_worked_example_r4():
    g = json.load(open(os.path.join(GOLDEN, "worked_r4.json")))
    q = np.array(g["q"], dtype=np.float64)
    keys = np.array(g["keys"], dtype=np.float64)
    # query at position 2 sees keys at positions 0, 1, 2 under the causal mask
    Q = np.stack([q, q, q])[None, :, None, :]
    K = keys[None, :, None, :]
    V = np.eye(3, 4)[None, :, None, :]  # v_j = e_j, so out_2 holds the three weights
    out, lse = oracle.attn_fwd(bf16(Q), bf16(K), bf16(V), window=-1, causal=True, rope_base=0.0, eps=-1.0)
    w = [float(x) for x in g["weights"]]
    np.testing.assert_allclose(out[0, 2, 0, :3], w, rtol=0, atol=1e-15)
    assert out[0, 2, 0, 3] == 0.0
    assert abs(lse[0, 0, 2] - float(g["lse"])) < 1e-15
    # the scores themselves: lse - log(weight) = max score; log-weights differ by score gaps
    s = np.log(out[0, 2, 0, :3]) + lse[0, 0, 2]
    np.testing.assert_allclose(s, g["scaled_scores"], atol=1e-14)
    # row 0 sees only k1: a single key gets weight 1 and lse = its score q.k1 / 2
    np.testing.assert_allclose(out[0, 0, 0], [1, 0, 0, 0], atol=0)
    assert abs(lse[0, 0, 0] - 0.5) < 1e-15
    P = oracle.attn_probs(bf16(Q), bf16(K), bf16(V), 0, 0, window=-1, causal=True, rope_base=0.0, eps=-1.0)
    np.testing.assert_allclose(P[2], w, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Normalisation and masks ("O que a Atenção Calcula": weights sum to 1; "A Máscara Causal")


@pytest.mark.parametrize("window,causal", [(-1, True), (3, True), (0, True), (2, False), (-1, False)])
def test_weights_sum_to_one_and_mask_zero(window, causal):
    T = 13
    q, k, v = make_qkv(1, T, 2, 16, seed=7)
    for h in range(2):
        P = oracle.attn_probs(q, k, v, 0, h, window=window, causal=causal)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        for i in range(T):
            for j in range(T):
                allowed = brute.visible(i, j, window, causal)
                assert (P[i, j] > 0) == allowed, (i, j)


def test_mask_literal_rows():
    """Literal visible sets written out by hand for T = 6."""
    T = 6
    q, k, v = make_qkv(1, T, 1, 8, seed=3)
    P = oracle.attn_probs(q, k, v, 0, 0, window=2, causal=True)
    assert [j for j in range(T) if P[4, j] > 0] == [2, 3, 4]
    assert [j for j in range(T) if P[0, j] > 0] == [0]
    assert [j for j in range(T) if P[1, j] > 0] == [0, 1]
    P = oracle.attn_probs(q, k, v, 0, 0, window=1, causal=False)
    assert [j for j in range(T) if P[3, j] > 0] == [2, 3, 4]
    assert [j for j in range(T) if P[5, j] > 0] == [4, 5]
    P = oracle.attn_probs(q, k, v, 0, 0, window=-1, causal=True)
    assert [j for j in range(T) if P[3, j] > 0] == [0, 1, 2, 3]
    P = oracle.attn_probs(q, k, v, 0, 0, window=0, causal=True)
    assert [j for j in range(T) if P[3, j] > 0] == [3]


@pytest.mark.parametrize("window,causal", [(-1, True), (4, True), (3, False)])
def test_masked_perturbation_invariance(window, causal):
    B, T, H, D = 1, 20, 2, 16
    q, k, v = make_qkv(B, T, H, D, seed=11)
    out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal)
    i = 9
    k2, v2 = k.clone(), v.clone()
    for j in range(T):
        if not brute.visible(i, j, window, causal):
            k2[:, j] = -k2[:, j] * 3
            v2[:, j] = v2[:, j] + 5
    out2, lse2 = oracle.attn_fwd(q, k2, v2, window=window, causal=causal)
    assert np.array_equal(out[:, i], out2[:, i])
    assert np.array_equal(lse[:, :, i], lse2[:, :, i])


@pytest.mark.parametrize("T", [1, 7, 64])
def test_window_ge_T_equals_full_causal(T):
    q, k, v = make_qkv(2, T, 3, 16, seed=5)
    ref_o, ref_l = oracle.attn_fwd(q, k, v, window=-1, causal=True)
    for w in (T - 1, T, T + 3, 10 * T):
        o, l = oracle.attn_fwd(q, k, v, window=w, causal=True)
        assert np.array_equal(o, ref_o) and np.array_equal(l, ref_l)
    if T > 2:
        o, _ = oracle.attn_fwd(q, k, v, window=T - 2, causal=True)
        assert not np.array_equal(o, ref_o)


def test_constant_v_gives_constant_out():
    B, T, H, D = 1, 33, 2, 16
    q, k, _ = make_qkv(B, T, H, D, seed=9)
    v = torch.full((B, T, H, D), 0.375, dtype=torch.bfloat16)
    for window, causal in [(-1, True), (5, True), (4, False)]:
        out, _ = oracle.attn_fwd(q, k, v, window=window, causal=causal)
        np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------------------------
# Closed form: q = 0 gives uniform weights over J(i), so lse = ln|J(i)| (pins the mask counts)


@pytest.mark.parametrize("window,causal,counts", [
    (2, True, [1, 2, 3, 3, 3, 3, 3, 3]),
    (0, True, [1] * 8),
    (-1, True, [1, 2, 3, 4, 5, 6, 7, 8]),
    (8, True, [1, 2, 3, 4, 5, 6, 7, 8]),
    (2, False, [3, 4, 5, 5, 5, 5, 4, 3]),
    (-1, False, [8] * 8),
    (0, False, [1] * 8),
])
def test_zero_query_closed_form(window, causal, counts):
    T, D = 8, 16
    _, k, v = make_qkv(1, T, 1, D, seed=13)
    q = torch.zeros((1, T, 1, D), dtype=torch.bfloat16)
    out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal, eps=1e-6)
    np.testing.assert_allclose(lse[0, 0], np.log(counts), rtol=0, atol=1e-15)
    vv = f64(v)[0, :, 0]
    lo_hi = [[j for j in range(T) if brute.visible(i, j, window, causal)] for i in range(T)]
    assert [len(x) for x in lo_hi] == counts
    for i in range(T):
        np.testing.assert_allclose(out[0, i, 0], vv[lo_hi[i]].mean(axis=0), rtol=0, atol=1e-14)


def test_zero_query_counts_large():
    """Sum over rows of exp(lse) = number of unmasked entries, at the workload's T and window."""
    T, D = 1024, 32
    _, k, v = make_qkv(1, T, 1, D, seed=17)
    q = torch.zeros((1, T, 1, D), dtype=torch.bfloat16)
    for window in (512, 1024, -1):
        _, lse = oracle.attn_fwd(q, k, v, window=window, causal=True)
        total = np.exp(lse[0, 0]).sum()
        assert abs(total - n_unmasked(T, window, True)) < 1e-6 * total
    # the figures quoted for one (b, h) pair of the T = 1024 workloads
    assert n_unmasked(1024, 512, True) == 393984
    assert n_unmasked(1024, 1024, True) == 524800


# ---------------------------------------------------------------------------------------------
# RMSNorm and RoPE (habr "Autoresearch" deep dive, train.py listing: norm, apply_rotary_emb)


def test_rmsnorm_values():
    x = bf16(np.array([3.0, 4.0]).reshape(1, 1, 1, 2))
    y = oracle.qk_prologue(x, rope_base=0.0, eps=0.0, round_qk=False)
    np.testing.assert_allclose(y.ravel(), [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-15)
    ones = bf16(np.ones((1, 1, 1, 8)))
    y = oracle.qk_prologue(ones, rope_base=0.0, eps=0.25, round_qk=False)
    np.testing.assert_allclose(y.ravel(), 1 / math.sqrt(1.25), rtol=1e-15)


def test_rmsnorm_identities():
    B, T, H, D = 2, 5, 3, 32
    x, _, _ = make_qkv(B, T, H, D, seed=21)
    eps = 0.3
    y = oracle.qk_prologue(x, rope_base=0.0, eps=eps, round_qk=False)
    xx = f64(x)
    ms = (xx ** 2).mean(-1)
    np.testing.assert_allclose((y ** 2).sum(-1), D * ms / (ms + eps), rtol=1e-13)
    # scale invariance with eps = 0 (2x is exact in bf16)
    y1 = oracle.qk_prologue(x, rope_base=0.0, eps=0.0, round_qk=False)
    y2 = oracle.qk_prologue((x.float() * 2).to(torch.bfloat16), rope_base=0.0, eps=0.0, round_qk=False)
    assert np.array_equal(y1, y2)


def test_rope_literal_values():
    """D = 4, base 10000: pair 0 is (x0, x2) at angle t, pair 1 is (x1, x3) at angle t/100."""
    tol = 1e-15

    def rot(vec, t):
        x = np.zeros((1, t + 1, 1, 4))
        x[0, t, 0] = vec
        return oracle.qk_prologue(bf16(x), rope_base=10000.0, eps=-1.0, round_qk=False)[0, t, 0]

    np.testing.assert_allclose(rot([1, 0, 0, 0], 1), [math.cos(1), 0, -math.sin(1), 0], atol=tol)
    np.testing.assert_allclose(rot([0, 0, 1, 0], 1), [math.sin(1), 0, math.cos(1), 0], atol=tol)
    np.testing.assert_allclose(rot([0, 1, 0, 0], 1), [0, math.cos(0.01), 0, -math.sin(0.01)], atol=tol)
    np.testing.assert_allclose(rot([0, 0, 0, 1], 3), [0, math.sin(0.03), 0, math.cos(0.03)], atol=tol)
    np.testing.assert_allclose(rot([0.5, -2, 1, 3], 0), [0.5, -2, 1, 3], atol=0)


def test_rope_norm_preserving_and_commutes_with_norm():
    B, T, H, D = 1, 40, 2, 64
    x, _, _ = make_qkv(B, T, H, D, seed=23)
    r = oracle.qk_prologue(x, rope_base=10000.0, eps=-1.0, round_qk=False)
    np.testing.assert_allclose((r ** 2).sum(-1), (f64(x) ** 2).sum(-1), rtol=1e-13)
    both = oracle.qk_prologue(x, rope_base=10000.0, eps=1e-6, round_qk=False)
    # normalise first, then rotate: apply RoPE to the normalised row by solving with the
    # rotation of the raw row (RoPE is linear, the norm is a per-row scale)
    ms = (f64(x) ** 2).mean(-1, keepdims=True)
    np.testing.assert_allclose(both, r / np.sqrt(ms + 1e-6), rtol=0, atol=1e-12)


def test_rope_relative_position():
    """With every q_t = a and every k_t = b, q_i . k_j depends only on i - j."""
    T, D = 24, 32
    a = np.random.default_rng(0).standard_normal(D)
    b = np.random.default_rng(1).standard_normal(D)
    qa = oracle.qk_prologue(bf16(np.tile(a, (1, T, 1, 1))), eps=1e-6, round_qk=False)[0, :, 0]
    kb = oracle.qk_prologue(bf16(np.tile(b, (1, T, 1, 1))), eps=1e-6, round_qk=False)[0, :, 0]
    S = qa @ kb.T
    for off in range(-T + 1, T):
        d = np.diagonal(S, offset=off)
        assert np.ptp(d) < 1e-11, off
    # and is not constant across offsets (positions do matter)
    assert np.ptp([np.diagonal(S, offset=o)[0] for o in range(-5, 6)]) > 1e-3


# ---------------------------------------------------------------------------------------------
# Special cases that reduce to library routines


@pytest.mark.parametrize("causal", [False, True])
def test_raw_mode_matches_scipy(causal):
    B, T, H, D = 1, 37, 2, 16
    q, k, v = make_qkv(B, T, H, D, seed=31)
    out, lse = oracle.attn_fwd(q, k, v, window=-1, causal=causal, rope_base=0.0, eps=-1.0)
    for h in range(H):
        Q, K, V = f64(q)[0, :, h], f64(k)[0, :, h], f64(v)[0, :, h]
        S = Q @ K.T / math.sqrt(D)
        if causal:
            S = np.where(np.tril(np.ones((T, T), dtype=bool)), S, -np.inf)
        np.testing.assert_allclose(out[0, :, h], scipy.special.softmax(S, axis=1) @ V, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, h], scipy.special.logsumexp(S, axis=1), rtol=0, atol=1e-13)


def test_round_bf16_matches_torch_and_brute():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                           [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3.3895e38]])
    f32 = vals.astype(np.float32).astype(np.float64)  # exactly representable in fp32
    ours = oracle.round_bf16(f32)
    ref = torch.tensor(f32.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    assert all(brute.round_bf16(float(a)) == b for a, b in zip(f32, ours))
    # ties go to the even neighbour
    assert oracle.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert oracle.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def test_round_qk_rounds_prologue_to_bf16():
    x, _, _ = make_qkv(1, 9, 2, 32, seed=41)
    a = oracle.qk_prologue(x, round_qk=True)
    b = oracle.qk_prologue(x, round_qk=False)
    assert np.array_equal(a, oracle.round_bf16(b))
    assert not np.array_equal(a, b)


# ---------------------------------------------------------------------------------------------
# Brute force for T <= 8 (every window, both mask modes, norm + RoPE on)


@pytest.mark.parametrize("T", range(1, 9))
def test_brute_force_small(T):
    B, H, D = 1, 2, 8
    q, k, v = make_qkv(B, T, H, D, seed=100 + T)
    qn, kn, vn = (f64(t).tolist() for t in (q, k, v))
    for window, causal in itertools.product(range(-1, 9), (True, False)):
        out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal)
        bo, bl = brute.forward(qn, kn, vn, window, causal, 10000.0, 1e-6)
        np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def test_brute_force_mask_counts():
    for T in range(1, 9):
        for window, causal in itertools.product(range(-1, 10), (True, False)):
            for i in range(T):
                assert n_allowed_keys(i, T, window, causal) == sum(brute.visible(i, j, window, causal)
                                                                    for j in range(T))


def test_rows_match_full():
    B, T, H, D = 2, 70, 3, 32
    q, k, v = make_qkv(B, T, H, D, seed=51)
    out, lse = oracle.attn_fwd(q, k, v, window=20, causal=True)
    rows = [(0, 0, 0), (1, 2, 69), (0, 1, 33), (1, 0, 21)]
    o, l = oracle.attn_rows(q, k, v, rows, window=20, causal=True)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(o[n], out[b, i, h], rtol=0, atol=1e-15)
        assert abs(l[n] - lse[b, h, i]) < 1e-15


# ---------------------------------------------------------------------------------------------
# Grouped K/V heads (habr "Autoresearch" deep dive, train.py listing: GPTConfig.n_kv_head and
# CausalSelfAttention, k and v with n_kv_head heads passed to the attention call): query head h
# reads K/V head h // (H // Hkv).


@pytest.mark.parametrize("H,Hkv,D,window,causal", [(4, 2, 32, 5, True), (4, 1, 64, -1, True),
                                                   (6, 3, 32, 3, False), (6, 2, 16, 11, True)])
def test_gqa_equals_mha_on_repeated_kv_heads(H, Hkv, D, window, causal):
    """Pinned to a library construction of the same attention: multi-head attention on K/V heads
    repeated with torch.repeat_interleave (head h of the result is head h // g of k). The two must
    agree bit for bit, for the full forward and for selected rows."""
    g = H // Hkv
    q, _, _ = make_qkv(2, 37, H, D, seed=900 + H)
    _, k, v = make_qkv(2, 37, Hkv, D, seed=901 + Hkv)
    out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal)
    ref, lref = oracle.attn_fwd(q, k.repeat_interleave(g, dim=2), v.repeat_interleave(g, dim=2),
                                window=window, causal=causal)
    assert np.array_equal(out, ref) and np.array_equal(lse, lref)
    rows = [(b, h, i) for b in (0, 1) for h in range(H) for i in (0, 6, 36)]
    ro, rl = oracle.attn_rows(q, k, v, rows, window=window, causal=causal)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(ro[n], out[b, i, h]) and rl[n] == lse[b, h, i]


def test_gqa_brute_force():
    """Brute force (pure Python) on K/V heads expanded by list indexing, T <= 6."""
    H, Hkv, D = 4, 2, 8
    for T in (1, 3, 6):
        q, _, _ = make_qkv(1, T, H, D, seed=910 + T)
        _, k, v = make_qkv(1, T, Hkv, D, seed=920 + T)
        qn, kn, vn = (f64(t).tolist() for t in (q, k, v))
        ke = [[[kn[b][t][h // (H // Hkv)] for h in range(H)] for t in range(T)] for b in range(1)]
        ve = [[[vn[b][t][h // (H // Hkv)] for h in range(H)] for t in range(T)] for b in range(1)]
        for window, causal in ((-1, True), (1, True), (2, False)):
            out, lse = oracle.attn_fwd(q, k, v, window=window, causal=causal)
            bo, bl = brute.forward(qn, ke, ve, window, causal, 10000.0, 1e-6)
            np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def test_gqa_rejects_non_divisor_heads():
    q, _, _ = make_qkv(1, 8, 4, 8, seed=1)
    _, k, v = make_qkv(1, 8, 3, 8, seed=2)
    with pytest.raises(AssertionError):
        oracle.attn_fwd(q, k, v)


# ---------------------------------------------------------------------------------------------
# Near ties of the bf16 rounding of q^, k^ (attn_oracle.c, steps 3 and 6). A single-precision
# evaluation of RoPE and the norm may round an element that lies within its error of a bf16
# midpoint the other way; the oracle's ambiguity radius must cover every such evaluation, and the
# slack it derives must bound every output that those choices lead to.

U = 2.0 ** -24


def _angles32(T, D, base):
    i = np.arange(D // 2, dtype=np.float64)
    th = np.arange(T, dtype=np.float64)[:, None] * np.power(base, -2.0 * i / D)[None, :]
    return np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)


def _fp32_variants(x, rope_base, eps):
    """Several single-precision evaluations of RoPE + norm of x [B, T, H, D] (float32 numpy, each
    operation rounded): the listing's order with numpy's pairwise sums; norm first with the scale
    folded into cos / sin; and a strictly sequential sum of squares from the last element down."""
    B, T, H, D = x.shape
    half = D // 2
    x = x.astype(np.float32)
    f = np.float32
    c, s = _angles32(T, D, rope_base) if rope_base > 0 else (None, None)
    c4 = None if c is None else c[None, :, None, :]
    s4 = None if s is None else s[None, :, None, :]
    e32 = f(eps)
    outs = []

    def rope(v):
        x1, x2 = v[..., :half], v[..., half:]
        return np.concatenate([x1 * c4 + x2 * s4, x2 * c4 - x1 * s4], axis=-1).astype(np.float32)

    # (a) listing order: rotate, then normalise
    y = rope(x) if rope_base > 0 else x.copy()
    if eps >= 0:
        ms = (y * y).sum(-1, keepdims=True, dtype=np.float32) / f(D)
        y = y * (f(1) / np.sqrt(ms + e32))
    outs.append(y.astype(np.float32))
    # (b) norm first, the scale folded into cos and sin
    r = np.ones(x.shape[:-1] + (1,), np.float32)
    if eps >= 0:
        ms = (x * x).sum(-1, keepdims=True, dtype=np.float32) * f(1.0 / D)
        r = (f(1) / np.sqrt(ms + e32)).astype(np.float32)
    if rope_base > 0:
        cr, sr = (c4 * r).astype(np.float32), (s4 * r).astype(np.float32)
        x1, x2 = x[..., :half], x[..., half:]
        y = np.concatenate([x1 * cr + x2 * sr, x2 * cr - x1 * sr], axis=-1)
    else:
        y = x * r
    outs.append(y.astype(np.float32))
    # (c) sequential sum of squares from the last element down, reciprocal square root last
    acc = np.zeros(x.shape[:-1], np.float32)
    for d in range(D - 1, -1, -1):
        acc = (acc + x[..., d] * x[..., d]).astype(np.float32)
    r = np.ones(x.shape[:-1] + (1,), np.float32)
    if eps >= 0:
        r = (f(1) / np.sqrt((acc / f(D) + e32).astype(np.float32)))[..., None].astype(np.float32)
    y = rope(x * r) if rope_base > 0 else x * r
    outs.append(y.astype(np.float32))
    return outs


@pytest.mark.parametrize("D,rope_base,eps", [(32, 10000.0, 1e-6), (64, 10000.0, 1e-6), (128, 10000.0, 1e-6),
                                             (64, 0.0, 1e-6), (64, 10000.0, -1.0), (64, 500.0, 0.3)])
def test_ambiguity_radius_covers_single_precision_evaluations(D, rope_base, eps):
    """Every single-precision evaluation rounds each element to a bf16 value within the oracle's
    ambiguity radius of the oracle's value; the radius is 0 for almost every element, and where an
    evaluation does round the other way the radius is positive."""
    x, _, _ = make_qkv(2, 512, 8, D, seed=61 + D)
    x = (x.float() * 3).to(torch.bfloat16)
    y, amb = oracle.qk_prologue(x, rope_base=rope_base, eps=eps, return_amb=True)
    flips = 0
    for y32 in _fp32_variants(f64(x), rope_base, eps):
        r32 = torch.tensor(y32).to(torch.bfloat16).double().numpy()
        dev = np.abs(r32 - y)
        assert (dev <= amb).all(), (dev - amb).max()
        flips += int((dev > 0).sum())
    assert flips > 0  # the evaluations do disagree with the double rounding somewhere
    assert 0 < (amb > 0).mean() < 0.02


def test_ambiguity_radius_literal_cases():
    """Exact small values (no RoPE, no norm) have no ambiguity; a value placed within the budget
    of a midpoint has a radius of one bf16 step, one placed outside it has none."""
    x = bf16(np.array([1.0, -2.5, 0.75, 3.0]).reshape(1, 1, 1, 4))
    y, amb = oracle.qk_prologue(x, rope_base=0.0, eps=-1.0, return_amb=True)
    assert np.array_equal(y.ravel(), [1.0, -2.5, 0.75, 3.0]) and not amb.any()
    # with the norm on: the row (1, 1/2, 1/2, 1/2) has mean square 7/16, so y = x r with
    # r = 1 / sqrt(7/16 + eps); choose eps so that y_0 = target, which for the target below sits
    # 2^-30 above the midpoint 1 + 2^-8 between 1 and 1 + 2^-7 (and y_1..3 = target / 2 the same
    # way above the midpoint 1/2 + 2^-9)
    row = bf16(np.array([1.0, 0.5, 0.5, 0.5]).reshape(1, 1, 1, 4))
    for offset, near in ((2.0 ** -30, True), (2.0 ** -14, False)):
        target = 1.0 + 2.0 ** -8 + offset
        y, amb = oracle.qk_prologue(row, rope_base=0.0, eps=1.0 / target ** 2 - 7.0 / 16.0, return_amb=True)
        assert np.array_equal(y.ravel(), [1 + 2.0 ** -7] + [0.5 + 2.0 ** -8] * 3)  # above the midpoints
        if near:  # within the evaluation budget of them: either neighbour is correct
            assert np.array_equal(amb.ravel(), [2.0 ** -7] + [2.0 ** -8] * 3)
        else:
            assert not amb.any()


def _brute_head(qh, kh, v, window, causal):
    """float64 softmax attention of one head from given q^, k^ (no prologue), v [T, D]."""
    T, D = qh.shape
    S = qh @ kh.T / math.sqrt(D)
    vis = np.array([[brute.visible(i, j, window, causal) for j in range(T)] for i in range(T)])
    S = np.where(vis, S, -np.inf)
    m = S.max(1, keepdims=True)
    w = np.exp(S - m)
    z = w.sum(1, keepdims=True)
    return (w / z) @ v, (m + np.log(z)).ravel()


@pytest.mark.parametrize("T,window,causal", [(1, -1, True), (4, -1, True), (6, 2, True), (5, 1, False),
                                             (8, -1, False)])
def test_slack_bounds_every_choice(T, window, causal):
    """Brute force: with the budget widened 2^8-fold (many ambiguous elements), every choice of
    q^, k^ within the radii, at the corners of the box and at random points inside it, gives
    outputs within the slack of the oracle's; and the slack is 0 for rows that no ambiguous
    element touches."""
    D, scale = 8, 2.0 ** 8
    rng = np.random.default_rng(T * 31 + window)
    q, k, v = make_qkv(1, T, 2, D, seed=700 + T)
    out, lse, os_, ls_ = oracle.attn_fwd(q, k, v, window=window, causal=causal, return_slack=True,
                                         amb_scale=scale)
    yq, aq = oracle.qk_prologue(q, return_amb=True, amb_scale=scale)
    yk, ak = oracle.qk_prologue(k, return_amb=True, amb_scale=scale)
    assert (aq > 0).any() and (ak > 0).any()
    vv = f64(v)
    for h in range(2):
        Q, K, AQ, AK, V = yq[0, :, h], yk[0, :, h], aq[0, :, h], ak[0, :, h], vv[0, :, h]
        o0, l0 = _brute_head(Q, K, V, window, causal)
        np.testing.assert_allclose(o0, out[0, :, h], atol=1e-13)
        worst_o, worst_l = np.zeros_like(o0), np.zeros_like(l0)
        for n in range(600):
            if n < 2:
                sq, sk = np.full(Q.shape, 1 - 2 * n), np.full(K.shape, 2 * n - 1)
            elif n < 300:
                sq, sk = rng.choice([-1.0, 0.0, 1.0], Q.shape), rng.choice([-1.0, 0.0, 1.0], K.shape)
            else:
                sq, sk = rng.uniform(-1, 1, Q.shape), rng.uniform(-1, 1, K.shape)
            o, l = _brute_head(Q + sq * AQ, K + sk * AK, V, window, causal)
            worst_o = np.maximum(worst_o, np.abs(o - o0))
            worst_l = np.maximum(worst_l, np.abs(l - l0))
        assert (worst_l <= ls_[0, h] + 1e-12).all(), (worst_l - ls_[0, h]).max()
        assert (worst_o <= os_[0, :, h] + 1e-12).all(), (worst_o - os_[0, :, h]).max()
        assert (ls_[0, h] > 0).any()


def test_slack_of_a_single_key_row_is_attained():
    """Row 0 under the causal mask sees one key, so its lse is the score q^_0 . k^_0 / sqrt(D) and
    its output is v_0: the lse slack equals the largest possible move of that score up to the
    second-order term, and the output slack is 0."""
    D, scale = 16, 2.0 ** 9
    for seed in range(5):
        q, k, v = make_qkv(1, 1, 1, D, seed=800 + seed)
        out, lse, os_, ls_ = oracle.attn_fwd(q, k, v, causal=True, return_slack=True, amb_scale=scale)
        yq, aq = oracle.qk_prologue(q, return_amb=True, amb_scale=scale)
        yk, ak = oracle.qk_prologue(k, return_amb=True, amb_scale=scale)
        Q, K, AQ, AK = yq.ravel(), yk.ravel(), aq.ravel(), ak.ravel()
        first = (AQ * np.abs(K) + np.abs(Q) * AK).sum() / math.sqrt(D)
        second = (AQ * AK).sum() / math.sqrt(D)
        assert first + second > 0
        # the corner with each perturbation aligned to the other factor's sign moves s by >= first - second
        best = ((Q + AQ * np.sign(K)) @ (K + AK * np.sign(Q)) - Q @ K) / math.sqrt(D)
        assert best >= first - second - 1e-15
        assert abs(ls_.item() - (first + second)) <= 1e-12 * max(1.0, first)
        assert os_.max() == 0.0


def test_slack_zero_without_rounding_or_ambiguity():
    q, k, v = make_qkv(1, 40, 2, 32, seed=905)
    _, _, os_, ls_ = oracle.attn_fwd(q, k, v, window=7, round_qk=False, return_slack=True)
    assert not os_.any() and not ls_.any()
    # raw mode on small integers: q^, k^ are the inputs themselves, exactly bf16
    qi, ki = (torch.randint(-3, 4, (1, 40, 2, 32)).to(torch.bfloat16) for _ in range(2))
    _, _, os_, ls_ = oracle.attn_fwd(qi, ki, v, rope_base=0.0, eps=-1.0, return_slack=True)
    assert not os_.any() and not ls_.any()
    # and the slack outputs leave out and lse unchanged
    a = oracle.attn_fwd(q, k, v, window=7)
    b = oracle.attn_fwd(q, k, v, window=7, return_slack=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    rows = [(0, 1, 39), (0, 0, 3)]
    ro, rl, ros, rls = oracle.attn_rows(q, k, v, rows, window=7, return_slack=True)
    for n, (bb, h, i) in enumerate(rows):
        assert np.array_equal(ro[n], b[0][bb, i, h]) and rl[n] == b[1][bb, h, i]
        assert np.array_equal(ros[n], b[2][bb, i, h]) and rls[n] == b[3][bb, h, i]


# ---------------------------------------------------------------------------------------------
# Value-embedding gate (NEXT-3; habr "Autoresearch" deep dive, train.py listing,
# CausalSelfAttention.forward, "Value Residual (ResFormer)"): v' = v + 2 sigmoid(x[..., :32] W^T) ve.


def _gate_inputs(seed, B=2, T=5, Hkv=3, D=8, C=32, w_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    bf = lambda *s, scale=1.0: (torch.randn(*s, generator=g) * scale).to(torch.bfloat16)
    return bf(B, T, Hkv, D), bf(B, T, Hkv, D), bf(B, T, C), bf(Hkv, C, scale=w_scale)


def test_value_gate_closed_forms():
    v, ve, x, w = _gate_inputs(1)
    vv, ee = f64(v), f64(ve)
    # zero gate weights: gate = 2 sigmoid(0) = 1 exactly, so v' = bf16(v + ve)
    got = oracle.value_gate(v, ve, x, torch.zeros_like(w))
    assert np.array_equal(got, oracle.round_bf16(vv + ee))
    # ve = 0 leaves v unchanged
    assert np.array_equal(oracle.value_gate(v, torch.zeros_like(ve), x, w), vv)
    # saturated logits: sum 32 * 4 = 128 -> sigmoid rounds to 1 (gate 2); -128 -> gate about 2e-56
    ones = torch.ones_like(x)
    got = oracle.value_gate(v, ve, ones, torch.full_like(w, 4.0))
    assert np.array_equal(got, oracle.round_bf16(vv + 2.0 * ee))
    got = oracle.value_gate(v, ve, ones, torch.full_like(w, -4.0))
    assert np.array_equal(got, vv)


def test_value_gate_matches_torch_bf16_evaluation():
    """The same expression evaluated by PyTorch on bf16 CPU tensors (each op rounds its result to
    bf16; the linear layer accumulates in fp32). The two agree wherever their gate logits agree;
    the logits differ by at most one bf16 step where fp32 accumulation rounds a near-tie the
    other way."""
    import torch.nn.functional as F

    v, ve, x, w = _gate_inputs(2, B=4, T=16, Hkv=4, D=16)
    got = oracle.value_gate(v, ve, x, w)
    logit_t = F.linear(x, w)  # bf16 [B, T, Hkv]
    gate_t = 2 * torch.sigmoid(logit_t)
    ref = (v + gate_t.unsqueeze(-1) * ve).to(torch.float64).numpy()
    xx, ww = f64(x), f64(w)
    logit_o = oracle.round_bf16(np.einsum("btc,hc->bth", xx, ww))
    same = logit_o == logit_t.to(torch.float64).numpy()
    assert same.mean() > 0.98
    step = np.abs(logit_o - logit_t.to(torch.float64).numpy())[~same]
    assert (step <= np.abs(logit_o[~same]) * 2.0 ** -7 + 1e-30).all()  # one bf16 step at most
    np.testing.assert_array_equal(got[same], ref[same])


def test_round_bf16_array_matches_the_scalar_routine():
    """The vectorised rounding against the C routine: random values over many binades, exact bf16
    values, midpoints (ties to even, both directions), values just either side of a midpoint."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(4000) * np.exp2(rng.integers(-60, 60, 4000))
    base = oracle.round_bf16_array(x)
    mids = base + np.sign(base) * np.abs(base) * 2.0 ** -9 * (1 + rng.integers(0, 2, 4000))
    cases = np.concatenate([x, base, mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf), [0.0, -0.0, 1.0,
                            1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -126, 3e38]])
    np.testing.assert_array_equal(oracle.round_bf16_array(cases), oracle.round_bf16(cases))


def _f32_value_gate(v, ve, x, w, order):
    """A single-precision evaluation of the gate: the logit summed in float32 in the given channel
    order, sigmoid via float32 exp, every listed step rounded to bf16 (torch)."""
    xx, ww = f64(x).astype(np.float32), f64(w).astype(np.float32)
    logit = np.zeros(xx.shape[:2] + (ww.shape[0],), dtype=np.float32)
    for c in order:
        logit = (logit + xx[:, :, None, c] * ww[None, None, :, c]).astype(np.float32)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
    lg = bf(logit)
    sig = bf((np.float32(1.0) / (np.float32(1.0) + np.exp(-lg).astype(np.float32))).astype(np.float32))
    prod = bf((2.0 * sig)[..., None] * f64(ve).astype(np.float32))
    return bf((f64(v).astype(np.float32) + prod).astype(np.float32)).astype(np.float64)


def test_value_gate_ambiguity_radius_covers_single_precision_evaluations():
    """Single-precision evaluations (channel orders forward, backward, random) land within the radius
    of the exact-then-rounded gate; the radius is zero on most rows and one bf16 step where nonzero."""
    v, ve, x, w = _gate_inputs(3, B=4, T=32, Hkv=4, D=16, w_scale=0.5)
    got, amb = oracle.value_gate(v, ve, x, w, return_amb=True)
    assert np.array_equal(got, oracle.value_gate(v, ve, x, w))
    rng = np.random.default_rng(1)
    for order in (range(32), range(31, -1, -1), rng.permutation(32)):
        alt = _f32_value_gate(v, ve, x, w, order)
        assert np.all(np.abs(alt - got) <= amb), np.max(np.abs(alt - got) - amb)
    zero_rows = (amb.max(axis=-1) == 0).mean()
    assert zero_rows > 0.8, zero_rows
    # a one-step change of the bf16 sigmoid moves the gate by at most 2^-7 of 2 and the product by that
    # much of |ve|, plus one bf16 step of v' for the roundings that follow
    nz = amb > 0
    assert np.all(amb[nz] <= np.abs(f64(ve))[nz] * 2.0 ** -6 + np.abs(got[nz]) * 2.0 ** -7)


def test_value_gate_ambiguity_radius_catches_a_forced_tie():
    """A row whose exact logit sits on a bf16 midpoint (1 + 2^-8, between 1 and 1 + 2^-7): the exact
    value rounds to even (1.0) and any evaluation error may move it up; the radius must show it."""
    B, T, Hkv, D, C = 1, 1, 1, 4, 32
    x = torch.zeros(B, T, C, dtype=torch.bfloat16)
    w = torch.zeros(Hkv, C, dtype=torch.bfloat16)
    x[0, 0, 0], w[0, 0] = 1.0, 1.0                    # 1
    x[0, 0, 1], w[0, 1] = 2.0 ** -8, 1.0              # + 2^-8: the midpoint
    v = torch.zeros(B, T, Hkv, D, dtype=torch.bfloat16)
    ve = torch.ones(B, T, Hkv, D, dtype=torch.bfloat16)
    got, amb = oracle.value_gate(v, ve, x, w, return_amb=True)
    assert (amb > 0).all()
