"""Shared helpers of the GPU parity tests: run the CUDA path through the binding, compare with
the oracle under the stated tolerances, and describe any mismatch."""
import numpy as np
import torch

OUT_ATOL = 2e-2   # max |out_gpu - out_oracle| on the bf16 output
LSE_RTOL = 1e-3   # |lse_gpu - lse_oracle| <= LSE_RTOL * max(1, |lse_oracle|)


def gpu_fwd(q, k, v, window=-1, causal=True, rope_base=10000.0, eps=1e-6, return_tensors=False):
    from sliding_window_attention_04_b300 import attn

    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = attn.attn_fwd(qd, kd, vd, window=window, causal=causal, rope_base=rope_base, eps=eps)
    torch.cuda.synchronize()
    st = attn.attn_device_status()
    assert st == 0, attn.status_string(st)
    if return_tensors:
        return out, lse
    return out.cpu().to(torch.float64).numpy(), lse.cpu().to(torch.float64).numpy()


def describe(out, ref, lse, lse_ref):
    err = np.abs(out - ref)
    idx = np.unravel_index(np.argmax(err), err.shape)
    lerr = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    lidx = np.unravel_index(np.argmax(lerr), lerr.shape)
    return (f"max|dout|={err.max():.3e} at {tuple(int(i) for i in idx)} (gpu {out[idx]:.5f} ref {ref[idx]:.5f}); "
            f"n>atol={int((err > OUT_ATOL).sum())}/{err.size}; "
            f"max lse err={lerr.max():.3e} at {tuple(int(i) for i in lidx)} "
            f"(gpu {lse[lidx]:.5f} ref {lse_ref[lidx]:.5f})")


def assert_close(out, ref, lse, lse_ref, what=""):
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    assert np.isfinite(lse).all(), f"{what}: non-finite lse"
    err = np.abs(out - ref).max() if out.size else 0.0
    lerr = (np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))).max() if lse.size else 0.0
    assert err <= OUT_ATOL and lerr <= LSE_RTOL, f"{what}: {describe(out, ref, lse, lse_ref)}"
    return err, lerr
