"""attn_fwd_noalloc: the forward call for callers that cannot allocate device memory.

Serving processes whose device memory is pre-divided by a framework allocator or a fixed pool,
and plug-in hosts that forbid libraries from allocating, cannot let the library cudaMalloc its
cos/sin table or error word. This entry point keeps those in a fixed device array of the
library instead. These tests call it through the C ABI and compare it with attn_fwd and with the
float64 oracle, within the tolerances of the parity tests, on two calls in a row (the second call
reuses the shared array with a different shape, so a stale table would show up); they also run it
at the exact size limit of that array and read its error word through attn_noalloc_status. This
file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import LSE_RTOL, OUT_ATOL, assert_close, oracle_fwd
from sliding_window_attention_04_b300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def _noalloc(attn, q, k, v, window, causal, rope_base, eps):
    B, T, H, D = q.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    rc = attn.attn_fwd_noalloc_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, H, T, D, window, int(causal), rope_base, eps,
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    return out, lse


def test_noalloc_matches_attn_fwd_and_oracle_on_two_calls_in_a_row():
    from sliding_window_attention_04_b300 import attn

    torch.cuda.set_device(0)
    attn.attn_init(0)  # only for the reference entry point; attn_fwd_noalloc does not need it
    cases = [((2, 300, 3, 64), 150, True, 10000.0, 1e-6, 11),
             ((1, 513, 2, 32), -1, True, 500.0, 1e-6, 12),
             ((1, 260, 2, 128), 100, True, 10000.0, 1e-6, 13)]
    for (B, T, H, D), window, causal, base, eps, seed in cases:
        qc, kc, vc = make_qkv(B, T, H, D, seed=seed)
        q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
        got_o, got_l = _noalloc(attn, q, k, v, window, causal, base, eps)
        ref_o, ref_l = attn.attn_fwd(q, k, v, window=window, causal=causal, rope_base=base, eps=eps)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_OK
        assert attn.attn_noalloc_status() == attn.ATTN_OK
        do = (got_o.double() - ref_o.double()).abs().max().item()
        dl = ((got_l.double() - ref_l.double()).abs() / ref_l.double().abs().clamp(min=1.0)).max().item()
        assert np.isfinite(do) and do <= OUT_ATOL, (T, D, do)
        assert np.isfinite(dl) and dl <= LSE_RTOL, (T, D, dl)
        ref, lref, os_, ls_ = oracle_fwd(qc, kc, vc, window=window, causal=causal, rope_base=base, eps=eps)
        assert_close(got_o.cpu().double().numpy(), ref, got_l.cpu().double().numpy(), lref,
                     f"noalloc T={T} D={D}", os_, ls_)


def test_noalloc_at_its_size_limit_and_beyond():
    """T * D / 2 = 524288 cos/sin pairs is the largest table the fixed array holds: that call runs
    (rows at the end of the sequence checked against the oracle); one position more is rejected."""
    import oracle
    from sliding_window_attention_04_b300 import attn

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    T, D = 16384, 64
    qc, kc, vc = make_qkv(1, T, 1, D, seed=17)
    q, k, v = qc.cuda(), kc.cuda(), vc.cuda()
    out, lse = _noalloc(attn, q, k, v, 4096, True, 10000.0, 1e-6)
    torch.cuda.synchronize()
    assert attn.attn_noalloc_status() == attn.ATTN_OK
    rows = np.array([(0, 0, i) for i in (0, 1, 8191, 12000, T - 129, T - 128, T - 2, T - 1)], dtype=np.int32)
    ref, lref, os_, ls_ = oracle.attn_rows(qc, kc, vc, rows, window=4096, causal=True, return_slack=True)
    o, l = out.cpu().double().numpy(), lse.cpu().double().numpy()
    assert_close(np.stack([o[0, i, 0] for _, _, i in rows]), ref, np.array([l[0, 0, i] for _, _, i in rows]), lref,
                 "noalloc T=16384 at the limit", os_, ls_)

    T2 = T + 1  # T * D / 2 = 524320 pairs, above the fixed 524288
    q2 = torch.zeros((1, T2, 1, D), dtype=torch.bfloat16, device="cuda")
    k2, v2, out2 = torch.zeros_like(q2), torch.zeros_like(q2), torch.empty_like(q2)
    lse2 = torch.empty((1, 1, T2), dtype=torch.float32, device="cuda")
    args = (q2.data_ptr(), k2.data_ptr(), v2.data_ptr(), out2.data_ptr(), lse2.data_ptr(), 1, 1, T2, D, 64, 1)
    assert attn.attn_fwd_noalloc_raw(*args, 10000.0, 1e-6, stream) == attn.ATTN_ERR_SCRATCH_LIMIT
    # without RoPE no table is needed, so the same shape runs
    assert attn.attn_fwd_noalloc_raw(*args, 0.0, 1e-6, stream) == attn.ATTN_OK
    torch.cuda.synchronize()
    assert torch.isfinite(out2.float()).all()
    assert attn.attn_noalloc_status() == attn.ATTN_OK


def test_noalloc_error_word_reports_a_timeout():
    """The bounded-wait self test writes the timeout code into attn_fwd_noalloc's error word (no
    fault involved); attn_noalloc_status reports it once, clears it, and later calls still work."""
    from sliding_window_attention_04_b300 import attn

    torch.cuda.set_device(0)
    assert attn.attn_noalloc_status() == attn.ATTN_OK
    assert attn.attn_noalloc_selftest_wait_timeout() == attn.ATTN_OK
    assert attn.attn_noalloc_status() == attn.ATTN_ERR_DEVICE_TIMEOUT
    assert attn.attn_noalloc_status() == attn.ATTN_OK
    qc, kc, vc = make_qkv(1, 200, 2, 64, seed=19)
    out, lse = _noalloc(attn, qc.cuda(), kc.cuda(), vc.cuda(), 64, True, 10000.0, 1e-6)
    torch.cuda.synchronize()
    assert attn.attn_noalloc_status() == attn.ATTN_OK
    ref, lref, os_, ls_ = oracle_fwd(qc, kc, vc, window=64, causal=True)
    assert_close(out.cpu().double().numpy(), ref, lse.cpu().double().numpy(), lref, "noalloc after timeout",
                 os_, ls_)
