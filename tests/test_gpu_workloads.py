"""The five workloads at full size, in the launch configuration the benchmark times.

For every distinct launch shape of the workloads, four complete (b, h) heads are compared with the
oracle element by element (the first head, the last head, one from the last group of heads the
persistent kernel's tickets hand out together, and one at random), plus sampled rows of other
heads; one ANDREA-12M layer is compared on every element. Properties that hold at any size are
checked on every output element. Tolerances and slack: gpu_helpers.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, gpu_fwd, oracle_fwd
from sliding_window_attention_04_b300 import configs
from sliding_window_attention_04_b300.inputs import layer_seed, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from sliding_window_attention_04_b300 import attn

    attn.attn_init(0)
    yield attn


def sample_rows(B, H, T, window, n, seed):
    """Random (b, h, i) rows plus the structurally interesting ones: first and last rows,
    both sides of every 128-row tile edge, and both sides of the window edge."""
    rng = np.random.default_rng(seed)
    special = {0, 1, 2, T - 1, T - 2}
    for e in range(128, T, 128):
        special |= {e - 1, e}
    if 0 < window < T:
        special |= {window - 1, window, window + 1, window + 127, window + 128}
    special = sorted(i for i in special if 0 <= i < T)
    rows = [(int(rng.integers(B)), int(rng.integers(H)), i) for i in special]
    rows += [(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(T))) for _ in range(n)]
    return np.array(rows, dtype=np.int32)


def check_sampled(q, k, v, layer, rope_base, eps, n, seed, what, out_t=None, lse_t=None):
    B, T, H, D = q.shape
    if out_t is None:
        out_t, lse_t = gpu_fwd(q, k, v, window=layer.window, causal=layer.causal, rope_base=rope_base, eps=eps,
                               return_tensors=True)
    # properties over every element: finite, and each output is a convex combination of v rows
    assert torch.isfinite(out_t).all() and torch.isfinite(lse_t).all(), what
    vmax = v.float().abs().amax(dim=1).cuda()  # [B, H_kv, D] max over positions
    vmax = vmax.repeat_interleave(H // v.shape[2], dim=1)  # query head h reads K/V head h // (H // H_kv)
    assert (out_t.float().abs() <= vmax[:, None] * (1 + 2 ** -7) + 1e-6).all(), what
    rows = sample_rows(B, H, T, layer.window, n, seed)
    ref, lref, os_, ls_ = oracle.attn_rows(q, k, v, rows, window=layer.window, causal=layer.causal,
                                           rope_base=rope_base, eps=eps, return_slack=True)
    out = out_t.cpu().to(torch.float64).numpy()
    lse = lse_t.cpu().to(torch.float64).numpy()
    got = np.stack([out[b, i, h] for b, h, i in rows])
    lgot = np.array([lse[b, h, i] for b, h, i in rows])
    return assert_close(got, ref, lgot, lref, what, os_, ls_)


def ticket_group_heads(B, H, Hkv, T, D):
    """Heads per group of the persistent kernel's tickets: as many (b, h) heads as have their K and V
    (2 T D bf16 values per K/V head, shared by H / Hkv query heads) within 64 MiB together."""
    per_head = 2 * T * D * 2 // (H // Hkv)
    return max(1, (64 << 20) // per_head)


def full_heads(B, H, Hkv, T, D, seed):
    """(b, h) heads compared in full: the first, the last, one from the last ticket group, one at random."""
    rng = np.random.default_rng(seed)
    hg = ticket_group_heads(B, H, Hkv, T, D)
    n_bh = B * H
    last_group_start = (n_bh - 1) // hg * hg
    picks = [0, n_bh - 1, int(rng.integers(last_group_start, n_bh)), int(rng.integers(n_bh))]
    out = []
    for bh in picks:
        if (bh // H, bh % H) not in out:
            out.append((bh // H, bh % H))
    return out


def check_full_heads(q, k, v, layer, rope_base, eps, seed, what, out_t, lse_t):
    B, T, H, D = q.shape
    Hkv = k.shape[2]
    out = out_t.cpu().to(torch.float64).numpy()
    lse = lse_t.cpu().to(torch.float64).numpy()
    for b, h in full_heads(B, H, Hkv, T, D, seed):
        hk = h // (H // Hkv)
        qs, ks, vs = (x[b:b + 1, :, hh:hh + 1].contiguous() for x, hh in ((q, h), (k, hk), (v, hk)))
        ref, lref, os_, ls_ = oracle_fwd(qs, ks, vs, window=layer.window, causal=layer.causal,
                                         rope_base=rope_base, eps=eps)
        assert_close(out[b:b + 1, :, h:h + 1], ref, lse[b:b + 1, h:h + 1], lref, f"{what} head ({b},{h})", os_, ls_)


def check_layer(q, k, v, layer, rope_base, eps, n, seed, what):
    """One full-size launch: every element checked for the properties, four complete heads and n
    sampled rows (plus the structural ones) against the oracle."""
    out_t, lse_t = gpu_fwd(q, k, v, window=layer.window, causal=layer.causal, rope_base=rope_base, eps=eps,
                           return_tensors=True)
    check_full_heads(q, k, v, layer, rope_base, eps, seed, what, out_t, lse_t)
    return check_sampled(q, k, v, layer, rope_base, eps, n, seed, what + " sampled", out_t, lse_t)


@pytest.mark.parametrize("widx", [1, 2, 3])
def test_andrea_workloads_sampled(widx):
    w = configs.workloads()[widx]
    seen = set()
    for li, layer in enumerate(w.layers):
        if (layer.window, layer.causal) in seen and li != len(w.layers) - 1:
            continue  # one S layer and the final L layer carry every distinct launch shape
        seen.add((layer.window, layer.causal))
        q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, li))
        check_layer(q, k, v, layer, w.rope_base, w.eps, 600, 1000 * widx + li, f"{w.name} layer {li}")


def test_andrea_12m_layer_full():
    """One S layer of the ANDREA-12M workload compared on every output element."""
    w = configs.workloads()[1]
    q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, 0))
    out, lse = gpu_fwd(q, k, v, window=w.layers[0].window, causal=True, rope_base=w.rope_base, eps=w.eps)
    ref, lref, os_, ls_ = oracle_fwd(q, k, v, window=w.layers[0].window, causal=True, rope_base=w.rope_base,
                                     eps=w.eps)
    assert_close(out, ref, lse, lref, "12M layer 0 full", os_, ls_)


@pytest.mark.parametrize("T", [1024, 2048, 4096, 8192])
def test_sweep_sampled(T):
    w = [x for x in configs.sweep_workloads() if x.T == T][0]
    for li, layer in enumerate(w.layers):
        q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, 10 * li + T // 1024))
        check_layer(q, k, v, layer, w.rope_base, w.eps, 300, T + li, f"{w.name} layer {li}")


@pytest.mark.parametrize("window", [1024, 2048])
def test_autoresearch_d128_shape_sampled(window):
    """The autoresearch default attention shape (habr "Autoresearch" deep dive, train.py listing:
    head_dim 128, sequence_len 2048; NEXT-2): B = 128, H = 4, T = 2048, D = 128, one S layer
    (W = T/2) and one full-causal layer, sampled rows against the oracle. This size runs many
    units per CTA through the D = 128 configuration's single Q slot."""
    from types import SimpleNamespace

    q, k, v = make_qkv(128, 2048, 4, 128, seed=7000 + window)
    layer = SimpleNamespace(window=window, causal=True)
    check_layer(q, k, v, layer, 10000.0, 1e-6, 300, 7100 + window, f"autoresearch D128 w={window}")


def test_gqa_shape_sampled():
    """Grouped K/V heads at a multi-wave size (H = 12 query heads over 4 K/V heads, D = 64)."""
    from types import SimpleNamespace

    q, _, _ = make_qkv(16, 1024, 12, 64, seed=7300)
    _, k, v = make_qkv(16, 1024, 4, 64, seed=7301)
    check_layer(q, k, v, SimpleNamespace(window=512, causal=True), 10000.0, 1e-6, 300, 7302, "gqa 12/4")
