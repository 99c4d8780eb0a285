"""attn_fwd_noalloc: the forward call for callers that cannot allocate device memory.

Serving processes whose device memory is pre-divided by a framework allocator or a fixed pool,
and plug-in hosts that forbid libraries from allocating, cannot let the library cudaMalloc its
cos/sin table or error word. This entry point keeps those in a fixed device array of the
library instead. These tests call it through the C ABI and compare it with attn_fwd, within the
tolerances of the parity tests, on two calls in a row (the second call reuses the shared array
with a different shape, so a stale table or error word would show up). This file is collected
last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import LSE_RTOL, OUT_ATOL
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


def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row():
    from sliding_window_attention_04_b300 import attn

    torch.cuda.set_device(0)
    attn.attn_init(0)  # only for the reference entry point; attn_fwd_noalloc does not need it
    cases = [((2, 300, 3, 64), 150, True, 10000.0, 1e-6, 11),
             ((1, 513, 2, 32), -1, True, 500.0, 1e-6, 12)]
    for (B, T, H, D), window, causal, base, eps, seed in cases:
        q, k, v = (t.cuda() for t in make_qkv(B, T, H, D, seed=seed))
        got_o, got_l = _noalloc(attn, q, k, v, window, causal, base, eps)
        ref_o, ref_l = attn.attn_fwd(q, k, v, window=window, causal=causal, rope_base=base, eps=eps)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == attn.ATTN_OK
        do = (got_o.double() - ref_o.double()).abs().max().item()
        dl = ((got_l.double() - ref_l.double()).abs() / ref_l.double().abs().clamp(min=1.0)).max().item()
        assert np.isfinite(do) and do <= OUT_ATOL, (T, D, do)
        assert np.isfinite(dl) and dl <= LSE_RTOL, (T, D, dl)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from sliding_window_attention_04_b300 import attn

    torch.cuda.set_device(0)
    T, D = 16385, 64  # T * D / 2 = 524320 cos/sin pairs, above the fixed 524288
    q = torch.zeros((1, T, 1, D), dtype=torch.bfloat16, device="cuda")
    k, v, out = torch.zeros_like(q), torch.zeros_like(q), torch.empty_like(q)
    lse = torch.empty((1, 1, T), dtype=torch.float32, device="cuda")
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), 1, 1, T, D, 64, 1)
    stream = torch.cuda.current_stream().cuda_stream
    assert attn.attn_fwd_noalloc_raw(*args, 10000.0, 1e-6, stream) == attn.ATTN_ERR_SCRATCH_LIMIT
    # without RoPE no table is needed, so the same shape runs
    assert attn.attn_fwd_noalloc_raw(*args, 0.0, 1e-6, stream) == attn.ATTN_OK
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
