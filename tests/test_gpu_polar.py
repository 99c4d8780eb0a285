"""GPU parity of the Polar Express orthogonalisation (include/polar.h) against the oracle.

Each product of every step is checked on its own: given the GPU's own input of that product (the
previous product's bf16 output), the GPU result must be the exact value rounded to bf16, except where
an fp32 evaluation may round the other way (oracle.polar_express.gemm_rounded reports that radius per
element). The normalisation likewise (normalize_rounded). The full call must equal the chain of its
steps bit for bit, and stay within the rounded chain's measured distance of the float64 iteration.
"""
import numpy as np
import pytest
import torch

from oracle import polar_express as pe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def polar():
    from sliding_window_attention_04_b300 import attn
    from sliding_window_attention_04_b300 import polar as p

    attn.attn_init(0)
    return p


def _f64(t):
    return t.detach().cpu().double().numpy()


def _within(name, got, ref, rad, mask=None):
    bad = np.abs(got - ref) > rad
    if mask is not None:
        bad &= mask
    assert not bad.any(), f"{name}: {int(bad.sum())} elements outside the radius, e.g. {np.argwhere(bad)[:3].tolist()}"


def _upper(s):
    """Elements of the 128 x 128 blocks on and above the diagonal (what the kernels store of A and B)."""
    blk = np.arange(s) // 128
    return blk[:, None] <= blk[None, :]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _check_end_to_end(name, full, g):
    """The full call against the oracle's chain at the bf16 rounding points (the same computation with every
    product rounded exactly): within 1 % of it (the two can differ only where a near-tie rounds the other
    way and the difference propagates), and no further from the float64 iteration than that chain plus 1 %
    (the chain itself drifts from the float64 iteration by one bf16 rounding per product: 2-5 % here)."""
    from test_oracle_polar import _rounded_chain

    chain = _rounded_chain(g)
    f64 = pe.polar_express(_f64(g))
    got = _f64(full)
    assert _rel(got, chain) < 1e-2, (name, _rel(got, chain))
    assert _rel(got, f64) <= _rel(chain, f64) + 1e-2, (name, _rel(got, f64), _rel(chain, f64))


def _sym(a):
    """The symmetric matrix the next product reads: stored blocks, and their mirrors below."""
    return np.where(_upper(a.shape[-1]), a, np.swapaxes(a, -1, -2))


SHAPES = [(2, 64, 96), (1, 96, 64), (3, 128, 128), (1, 72, 200), (1, 200, 72), (2, 256, 384), (1, 384, 256),
          (1, 8, 8), (2, 8, 264), (1, 264, 8), (1, 136, 392)]


@pytest.mark.parametrize("batch,m,n", SHAPES)
def test_every_product_matches_the_rounded_oracle(polar, batch, m, n):
    g = torch.randn(batch, m, n, generator=torch.Generator().manual_seed(m * 1000 + n)).to(torch.bfloat16)
    x = polar.normalize(g.cuda())
    torch.cuda.synchronize()
    ref, rad = pe.normalize_rounded(g)
    _within("normalize", _f64(x), ref, rad)
    tall = m > n
    for k, (a, b, c) in enumerate(pe.POLAR_EXPRESS_COEFFS):
        y, A, B = polar.step(x, k)
        torch.cuda.synchronize()
        xh, Ah, Bh, yh = _f64(x), _f64(A), _f64(B), _f64(y)
        up = _upper(Ah.shape[-1])
        Ah, Bh = _sym(Ah), _sym(Bh)
        xt = np.swapaxes(xh, -1, -2)
        Aref, ra = pe.gemm_rounded(xt, xh) if tall else pe.gemm_rounded(xh, xt)
        _within(f"step {k} A", Ah, Aref, ra, up)
        Bref, rb = pe.gemm_rounded(Ah, Ah, c, b, Ah)
        _within(f"step {k} B", Bh, Bref, rb, up)
        Yref, ry = pe.gemm_rounded(xh, Bh, 1.0, a, xh) if tall else pe.gemm_rounded(Bh, xh, 1.0, a, xh)
        _within(f"step {k} X", yh, Yref, ry)
        x = y.clone()
    full = polar.polar_express(g.cuda())
    torch.cuda.synchronize()
    assert torch.equal(full, x)
    _check_end_to_end(f"{batch}x{m}x{n}", full, g)


def test_model_shaped_batches(polar):
    """Muon's groups of the ANDREA-120M shape at the batch sizes the bench times (48 x 768 x 768, 12 x 768 x
    3072 wide, 12 x 3072 x 768 tall): the last step's product over the whole batch against the rounded
    oracle on the GPU's own inputs of that step, the full call equal to its steps, and the end-to-end
    check on four matrices of each batch."""
    for batch, m, n in ((48, 768, 768), (12, 768, 3072), (12, 3072, 768)):
        g = torch.randn(batch, m, n, generator=torch.Generator().manual_seed(m + n)).to(torch.bfloat16)
        gc = g.cuda()
        full = polar.polar_express(gc)
        x4 = polar.normalize(gc)
        for k in range(4):
            x4, _, _ = polar.step(x4, k)
            x4 = x4.clone()
        y, A, B = polar.step(x4, 4)
        torch.cuda.synchronize()
        assert torch.equal(y, full)
        a, b, c = pe.POLAR_EXPRESS_COEFFS[4]
        xh, Ah, Bh = _f64(x4), _sym(_f64(A)), _sym(_f64(B))
        tall = m > n
        Yref, ry = pe.gemm_rounded(xh, Bh, 1.0, a, xh) if tall else pe.gemm_rounded(Bh, xh, 1.0, a, xh)
        _within(f"{m}x{n} last step", _f64(y), Yref, ry)
        # every matrix of a batch is computed independently: the end-to-end check samples a few of them
        k = 4 if batch >= 4 else batch
        _check_end_to_end(f"{batch}x{m}x{n}", full[:k], g[:k])


def test_normalize_in_place_and_many_chunks(polar):
    """In place equals out of place; a 2048 x 8192 matrix spans 1024 chunks of the two-pass sum and still
    lies within the rounded oracle's radius; two calls agree bit for bit."""
    g = torch.randn(3, 200, 72, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16).cuda()
    ref = polar.normalize(g)
    h = g.clone()
    polar.normalize(h, out=h)
    torch.cuda.synchronize()
    assert torch.equal(h, ref)
    big = (torch.randn(1, 2048, 8192, generator=torch.Generator().manual_seed(10)) * 3.0).to(torch.bfloat16)
    x1 = polar.normalize(big.cuda())
    x2 = polar.normalize(big.cuda())
    torch.cuda.synchronize()
    assert torch.equal(x1, x2)
    r, rad = pe.normalize_rounded(big)
    _within("normalize 2048x8192", _f64(x1), r, rad)


def test_executed_flop_count(polar):
    """One 128 x 128 block: every product is computed in full (the listing's 6 s^3); larger matrices
    skip the blocks of A and B below the diagonal, so fewer than the listing's count but more than the
    full Y product alone."""
    assert polar.step_flops(1, 128, 128) == 6 * 128 ** 3
    s, l = 768, 3072
    for bt, m, n in ((48, s, s), (12, s, l), (12, l, s)):
        listing = bt * (4 * s * s * max(m, n) + 2 * s ** 3)
        y_only = bt * 2 * s * m * n
        assert y_only < polar.step_flops(bt, m, n) < listing
