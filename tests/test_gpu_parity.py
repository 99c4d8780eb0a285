"""Parity of the CUDA path (through the C ABI) with the float64 oracle on the same seeded inputs.

Tolerances: max |out - oracle| <= 2e-2 on the bf16 output; |lse - oracle| <= 1e-3 * max(1, |lse|),
each widened by the oracle's near-tie slack of that element (gpu_helpers).
"""
import itertools

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, gpu_fwd, oracle_fwd
from sliding_window_attention_04_b300 import configs
from sliding_window_attention_04_b300.inputs import layer_seed, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from sliding_window_attention_04_b300 import attn

    attn.attn_init(0)
    yield attn


def check(q, k, v, window, causal, rope_base=10000.0, eps=1e-6, what=""):
    out, lse = gpu_fwd(q, k, v, window=window, causal=causal, rope_base=rope_base, eps=eps)
    ref, lref, os_, ls_ = oracle_fwd(q, k, v, window=window, causal=causal, rope_base=rope_base, eps=eps)
    return assert_close(out, ref, lse, lref, what or f"w={window} c={causal}", os_, ls_)


def test_tiny_workload_full():
    w = configs.workloads()[0]
    q, k, v = make_qkv(w.B, w.T, w.H, w.D, seed=layer_seed(w.index, 0))
    check(q, k, v, w.layers[0].window, True, w.rope_base, w.eps, "tiny")


@pytest.mark.parametrize("D", [32, 64, 128])
def test_brute_force_shapes(D):
    """Every T <= 8, every window -1..8, both mask modes (oracle pinned to brute force there)."""
    for T in range(1, 9):
        q, k, v = make_qkv(1, T, 2, D, seed=500 + T)
        for window, causal in itertools.product(range(-1, 9), (True, False)):
            check(q, k, v, window, causal, what=f"T={T} D={D} w={window} c={causal}")


CASES = [(-1, True), (0, True), (1, True), (127, True), (128, True), (200, True), ("half", True),
         (-1, False), (0, False), (100, False)]


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("T", [129, 300, 513])
def test_ragged_multitile(D, T):
    q, k, v = make_qkv(2, T, 3, D, seed=7 * T + D)
    for window, causal in CASES:
        wnd = T // 2 if window == "half" else window
        check(q, k, v, wnd, causal, what=f"T={T} D={D} w={wnd} c={causal}")


def test_worked_example_r4_gpu():
    """The worked R^4 example ("geometry_of_andrea", "Lendo uma Projeção") at D = 64: zero-padded
    and q scaled by sqrt(64/4) = 4 so that q.k / sqrt(64) reproduces the scores 0.5, 0.5, 0."""
    D = 64
    q = torch.zeros((1, 3, 1, D))
    q[0, :, 0, 0] = 4.0
    q[0, :, 0, 2] = 4.0
    k = torch.zeros((1, 3, 1, D))
    k[0, 0, 0, 0] = 1.0
    k[0, 1, 0, 2] = 1.0
    k[0, 2, 0, 1] = 1.0
    k[0, 2, 0, 3] = 1.0
    v = torch.zeros((1, 3, 1, D))
    for j in range(3):
        v[0, j, 0, j] = 1.0
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    out, lse = gpu_fwd(q, k, v, window=-1, causal=True, rope_base=0.0, eps=-1.0)
    w = [0.38365173119055069, 0.38365173119055069, 0.23269653761889861]
    np.testing.assert_allclose(out[0, 2, 0, :3], w, atol=4e-3)
    assert abs(lse[0, 0, 2] - 1.4580200879470337) < 1e-3
    assert abs(lse[0, 0, 0] - 0.5) < 1e-3


@pytest.mark.parametrize("rope_base,eps", [(0.0, 1e-6), (10000.0, -1.0), (0.0, -1.0), (500.0, 0.1)])
def test_prologue_modes(rope_base, eps):
    q, k, v = make_qkv(1, 300, 2, 64, seed=77)
    if eps < 0:  # without the norm, keep raw scores in a sane range
        q = (q.float() * 0.25).to(torch.bfloat16)
    check(q, k, v, 100, True, rope_base=rope_base, eps=eps, what=f"base={rope_base} eps={eps}")


@pytest.mark.parametrize("D", [32, 64, 128])
def test_masked_perturbation_bitwise(D):
    T, window = 400, 150
    q, k, v = make_qkv(1, T, 2, D, seed=91)
    out, lse = gpu_fwd(q, k, v, window=window, causal=True)
    i = 260
    k2, v2 = k.clone(), v.clone()
    masked = [j for j in range(T) if j > i or j < i - window]
    k2[:, masked] = (-3 * k2[:, masked].float()).to(torch.bfloat16)
    v2[:, masked] = (v2[:, masked].float() + 5).to(torch.bfloat16)
    out2, lse2 = gpu_fwd(q, k2, v2, window=window, causal=True)
    assert np.array_equal(out[:, i], out2[:, i])
    assert np.array_equal(lse[:, :, i], lse2[:, :, i])
    assert not np.array_equal(out[:, T - 1], out2[:, T - 1])


@pytest.mark.parametrize("T", [1, 200, 256])
def test_window_ge_T_bitwise_equals_causal(T):
    q, k, v = make_qkv(2, T, 2, 64, seed=13)
    ref = gpu_fwd(q, k, v, window=-1, causal=True)
    for w in (T - 1, T, 5 * T):
        got = gpu_fwd(q, k, v, window=w, causal=True)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), w


def test_deterministic():
    q, k, v = make_qkv(2, 700, 3, 64, seed=3)
    a = gpu_fwd(q, k, v, window=300, causal=True)
    b = gpu_fwd(q, k, v, window=300, causal=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_constant_v():
    q, k, _ = make_qkv(1, 333, 4, 64, seed=5)
    v = torch.full((1, 333, 4, 64), 0.6875, dtype=torch.bfloat16)
    out, _ = gpu_fwd(q, k, v, window=100, causal=True)
    # the weights are rounded to bf16 for P.V while the normaliser sums them in fp32, so the
    # result may land on a neighbouring bf16 value: at most one ulp (2^-8 in [0.5, 1))
    assert np.abs(out - 0.6875).max() <= 2 ** -8


def test_zero_query_closed_form_gpu():
    """q = 0 gives uniform weights over the visible keys: lse = ln|J(i)| (pins the mask counts)."""
    T = 1000
    _, k, v = make_qkv(1, T, 2, 64, seed=19)
    q = torch.zeros_like(k)
    for window, causal in [(512, True), (-1, True), (0, True), (37, False)]:
        _, lse = gpu_fwd(q, k, v, window=window, causal=causal)
        counts = np.array([configs.n_allowed_keys(i, T, window, causal) for i in range(T)])
        np.testing.assert_allclose(lse[0, 0], np.log(counts), atol=1e-4)


def test_lse_optional_and_streams():
    from sliding_window_attention_04_b300 import attn

    q, k, v = (t.cuda() for t in make_qkv(1, 300, 2, 32, seed=23))
    o1, l1 = attn.attn_fwd(q, k, v, window=64)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = attn.attn_fwd(q, k, v, window=64, return_lse=False)
    s.synchronize()
    torch.cuda.synchronize()
    assert l2 is None
    assert torch.equal(o1, o2)


def test_gpu_error_paths():
    from sliding_window_attention_04_b300 import attn

    x = torch.zeros((1, 8, 1, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(x, x, x)
    assert e.value.code == attn.ATTN_ERR_UNSUPPORTED
    y = torch.zeros((1, 8, 1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(y, y, y, out=y)  # out aliases q
    assert e.value.code == attn.ATTN_ERR_INVALID_ARG


def test_bounded_wait_reports_timeout_and_context_survives():
    from sliding_window_attention_04_b300 import attn

    assert attn.attn_device_status() == attn.ATTN_OK
    attn.attn_selftest_wait_timeout()
    assert attn.attn_device_status() == attn.ATTN_ERR_DEVICE_TIMEOUT
    assert attn.attn_device_status() == attn.ATTN_OK  # cleared by the read
    check(*make_qkv(1, 256, 2, 64, seed=29), 128, True, what="after timeout self-test")


def test_destroy_and_reinit():
    from sliding_window_attention_04_b300 import attn

    q, k, v = (t.cuda() for t in make_qkv(1, 64, 1, 64, seed=31))
    o1, _ = attn.attn_fwd(q, k, v)
    attn.attn_destroy()
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(q, k, v)
    assert e.value.code == attn.ATTN_ERR_NOT_INITIALIZED
    attn.attn_init(0)
    o2, _ = attn.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_fast_kernel_is_used_for_every_head_dim():
    from sliding_window_attention_04_b300 import attn

    assert attn.attn_fwd_kernel(32) == "ws"
    assert attn.attn_fwd_kernel(64) == "ws"
    assert attn.attn_fwd_kernel(128) == "ws"


def test_many_calls_reuse_ticket_slots():
    """More calls than the persistent kernel has ticket-counter slots (256), back to back on one
    stream, then on two streams in turn: every result must be bit-identical to the first."""
    from sliding_window_attention_04_b300 import attn

    q, k, v = (t.cuda() for t in make_qkv(3, 600, 5, 64, seed=41))
    ref, lref = attn.attn_fwd(q, k, v, window=200)
    outs = [attn.attn_fwd(q, k, v, window=200) for _ in range(300)]
    s2 = torch.cuda.Stream()
    for i in range(40):
        s = s2 if i % 2 else torch.cuda.current_stream()
        s.wait_stream(torch.cuda.current_stream() if i % 2 else s2)
        with torch.cuda.stream(s):
            outs.append(attn.attn_fwd(q, k, v, window=200))
    torch.cuda.synchronize()
    assert attn.attn_device_status() == attn.ATTN_OK
    for o, l in outs:
        assert torch.equal(o, ref) and torch.equal(l, lref)
    out, lse = ref.cpu().double().numpy(), lref.cpu().double().numpy()
    r, lr, os_, ls_ = oracle_fwd(q.cpu(), k.cpu(), v.cpu(), window=200, causal=True)
    assert_close(out, r, lse, lr, "many calls", os_, ls_)


@pytest.mark.parametrize("D,H,Hkv,T,window", [(64, 4, 2, 513, 127), (64, 6, 1, 300, -1), (32, 4, 2, 300, 100),
                                             (128, 4, 2, 256, 64), (64, 8, 2, 1024, 512)])
def test_gqa_parity(D, H, Hkv, T, window):
    """Grouped K/V heads (k, v with Hkv heads; query head h reads K/V head h // (H // Hkv))."""
    q, _, _ = make_qkv(2, T, H, D, seed=31 * T + H)
    _, k, v = make_qkv(2, T, Hkv, D, seed=37 * T + Hkv)
    check(q, k, v, window, True, what=f"gqa D={D} H={H} Hkv={Hkv} T={T} w={window}")


@pytest.mark.parametrize("D", [32, 64, 128])
def test_gqa_bitwise_equals_repeated_heads(D):
    """The grouped call computes exactly what the multi-head call computes on repeated K/V heads."""
    H, Hkv, T = 6, 2, 400
    q, _, _ = make_qkv(1, T, H, D, seed=4242)
    _, k, v = make_qkv(1, T, Hkv, D, seed=4343)
    out, lse = gpu_fwd(q, k, v, window=150, causal=True, return_tensors=True)
    ref, lref = gpu_fwd(q, k.repeat_interleave(H // Hkv, dim=2), v.repeat_interleave(H // Hkv, dim=2), window=150,
                        causal=True, return_tensors=True)
    assert torch.equal(out, ref) and torch.equal(lse, lref)
