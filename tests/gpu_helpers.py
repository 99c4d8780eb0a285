"""Shared helpers of the GPU parity tests: run the CUDA path through the binding, compare it with
the float64 oracle under the stated tolerances, and describe any mismatch.

Tolerances: max |out - oracle| <= 2e-2 on the bf16 output and |lse - oracle| <= 1e-3 * max(1, |lse|),
each widened by the oracle's slack for that element. The slack is 0 unless an element of q^ or k^
lies so close to a bf16 rounding midpoint that a single-precision evaluation of RoPE and the norm
may round it either way (both are correct); it bounds how far those choices can move the output
(attn_oracle.c, steps 3 and 6). Every comparison records how much slack it used; the session
prints a table of it at the end.
"""
import numpy as np
import torch

OUT_ATOL = 2e-2   # max |out_gpu - out_oracle| on the bf16 output
LSE_RTOL = 1e-3   # |lse_gpu - lse_oracle| <= LSE_RTOL * max(1, |lse_oracle|)

# one entry per comparison: (what, rows, rows with slack > 0, max lse slack, max out slack,
# rows that needed their slack to pass, max |dout|, max scaled lse error)
SLACK_LOG = []


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


def oracle_fwd(q, k, v, **kw):
    """The oracle's (out, lse, out_slack, lse_slack) for the same call."""
    import oracle

    return oracle.attn_fwd(q, k, v, return_slack=True, **kw)


def describe(out, ref, lse, lse_ref, tol_out, tol_lse):
    err = np.abs(out - ref)
    idx = np.unravel_index(np.argmax(err - tol_out), err.shape)
    lerr = np.abs(lse - lse_ref)
    lidx = np.unravel_index(np.argmax(lerr - tol_lse), lerr.shape)
    return (f"worst out at {tuple(int(i) for i in idx)}: gpu {out[idx]:.5f} ref {ref[idx]:.5f} "
            f"(|d| {err[idx]:.3e} vs tol {np.broadcast_to(tol_out, err.shape)[idx]:.3e}); "
            f"n>tol={int((err > tol_out).sum())}/{err.size}; "
            f"worst lse at {tuple(int(i) for i in lidx)}: gpu {lse[lidx]:.5f} ref {lse_ref[lidx]:.5f} "
            f"(|d| {lerr[lidx]:.3e} vs tol {np.broadcast_to(tol_lse, lerr.shape)[lidx]:.3e})")


def assert_close(out, ref, lse, lse_ref, what="", out_slack=None, lse_slack=None):
    """out/ref [..., D] and lse/lse_ref [...] (rows in the same order: [B, T, H, D] with [B, H, T],
    or [n, D] with [n]); slacks shaped like ref and lse_ref (None: 0)."""
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    assert np.isfinite(lse).all(), f"{what}: non-finite lse"
    out_slack = np.zeros_like(ref) if out_slack is None else out_slack
    lse_slack = np.zeros_like(lse_ref) if lse_slack is None else lse_slack
    tol_out = OUT_ATOL + out_slack
    tol_lse = LSE_RTOL * np.maximum(1.0, np.abs(lse_ref)) + lse_slack
    err = np.abs(out - ref)
    lerr = np.abs(lse - lse_ref)
    ok = (err <= tol_out).all() and (lerr <= tol_lse).all()
    # rows that pass only thanks to their slack (the near-tie choices of the kernel differed)
    needed = int((lerr > LSE_RTOL * np.maximum(1.0, np.abs(lse_ref))).sum())
    needed_out = int((err.reshape(-1, err.shape[-1]) > OUT_ATOL).any(-1).sum()) if err.size else 0
    SLACK_LOG.append((what, int(lse_ref.size), int((lse_slack > 0).sum()), float(lse_slack.max(initial=0.0)),
                      float(out_slack.max(initial=0.0)), needed + needed_out,
                      float(err.max(initial=0.0)),
                      float((lerr / np.maximum(1.0, np.abs(lse_ref))).max(initial=0.0))))
    assert ok, f"{what}: {describe(out, ref, lse, lse_ref, tol_out, tol_lse)}"
    return float(err.max(initial=0.0)), float((lerr / np.maximum(1.0, np.abs(lse_ref))).max(initial=0.0))


def slack_table():
    """Lines of the per-comparison slack report."""
    if not SLACK_LOG:
        return []
    lines = ["parity slack per comparison (rows | rows with slack | max lse slack | max out slack | "
             "rows that needed slack | max |dout| | max lse err / max(1,|lse|)):"]
    for what, rows, nsl, mls, mos, need, dout, dl in SLACK_LOG:
        lines.append(f"  {what}: {rows} | {nsl} | {mls:.2e} | {mos:.2e} | {need} | {dout:.2e} | {dl:.2e}")
    tot = sum(r[1] for r in SLACK_LOG)
    lines.append(f"  total: {len(SLACK_LOG)} comparisons, {tot} rows, {sum(r[2] for r in SLACK_LOG)} with slack, "
                 f"{sum(r[5] for r in SLACK_LOG)} needed it; max lse slack "
                 f"{max(r[3] for r in SLACK_LOG):.2e}, max out slack {max(r[4] for r in SLACK_LOG):.2e}")
    return lines
