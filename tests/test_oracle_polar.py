"""Pins of the Polar Express oracle (oracle/polar_express.py), CPU only."""
import numpy as np
import pytest

from oracle import polar_express as pe


def _spectral(g, steps):
    """The same map computed through numpy's SVD: normalise, then apply each step's odd polynomial
    a s + b s^3 + c s^5 to the singular values, keeping the singular vectors."""
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    s = s / (np.sqrt(np.sum(g * g)) * 1.02 + 1e-6)
    for a, b, c in pe.POLAR_EXPRESS_COEFFS[:steps]:
        s = a * s + b * s ** 3 + c * s ** 5
    return (u * s[..., None, :]) @ vt


@pytest.mark.parametrize("m,n", [(16, 16), (24, 8), (8, 24), (64, 48)])
@pytest.mark.parametrize("steps", [1, 3, 5])
def test_iteration_equals_polynomial_on_singular_values(m, n, steps):
    g = np.random.default_rng(m * 100 + n).standard_normal((m, n))
    np.testing.assert_allclose(pe.polar_express(g, steps), _spectral(g, steps), rtol=0, atol=1e-10)


def test_wide_form_is_the_transpose_of_the_tall_form():
    g = np.random.default_rng(3).standard_normal((40, 12))
    np.testing.assert_allclose(pe.polar_express(g.T), pe.polar_express(g).T, rtol=0, atol=1e-12)


def test_batched_matrices_are_independent():
    g = np.random.default_rng(4).standard_normal((3, 20, 10))
    got = pe.polar_express(g)
    for i in range(3):
        np.testing.assert_allclose(got[i], pe.polar_express(g[i]), rtol=0, atol=1e-13)


def test_close_to_the_polar_factor_for_well_conditioned_input():
    """Singular values in [0.5, 1] (times a scale): after five steps every one ends near 1, so the
    result is near U V^T."""
    rng = np.random.default_rng(5)
    u, _ = np.linalg.qr(rng.standard_normal((32, 32)))
    v, _ = np.linalg.qr(rng.standard_normal((32, 32)))
    s = np.linspace(0.5, 1.0, 32) * 7.0
    g = (u * s) @ v.T
    got = pe.polar_express(g)
    sv = np.linalg.svd(got, compute_uv=False)
    assert sv.min() > 0.85 and sv.max() < 1.15, (sv.min(), sv.max())
    assert np.abs(got - u @ v.T).max() < 0.15


import torch  # noqa: E402


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def test_gemm_rounded_exact_on_small_integers():
    rng = np.random.default_rng(8)
    p = rng.integers(-2, 3, (2, 5, 4)).astype(np.float64)
    q = rng.integers(-2, 3, (2, 4, 6)).astype(np.float64)
    r = rng.integers(-3, 4, (2, 5, 6)).astype(np.float64)
    d, rad = pe.gemm_rounded(p, q, 2.0, -1.0, r)
    np.testing.assert_array_equal(d, 2.0 * (p @ q) - r)
    # exact results away from zero have no other rounding; at exact zeros the radius is the tiny budget
    assert not rad[d != 0].any() and rad.max() < 1e-4


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (15.878769915207462, -22.48329292557795), (1.0, 2.3465413258596377)])
def test_gemm_rounded_radius_covers_float32_evaluations(alpha, beta):
    rng = np.random.default_rng(9)
    p, q, r = (_bf16(rng.standard_normal(s) * 0.3) for s in ((2, 24, 40), (2, 40, 16), (2, 24, 16)))
    d, rad = pe.gemm_rounded(p, q, alpha, beta, r)
    a32, b32 = np.float32(alpha), np.float32(beta)
    for order in (range(40), range(39, -1, -1)):
        acc = np.zeros((2, 24, 16), dtype=np.float32)
        for k in order:
            acc = (acc + p[:, :, k:k + 1].astype(np.float32) * q[:, k:k + 1, :].astype(np.float32)).astype(np.float32)
        out = _bf16((a32 * acc + b32 * r.astype(np.float32)).astype(np.float32))
        assert np.all(np.abs(out - d) <= rad), np.max(np.abs(out - d) - rad)


def test_normalize_rounded_radius_covers_float32_and_exact_case():
    rng = np.random.default_rng(10)
    g = _bf16(rng.standard_normal((3, 16, 32)))
    x, rad = pe.normalize_rounded(g)
    g32 = g.astype(np.float32)
    ss = np.zeros((3, 1, 1), dtype=np.float32)
    for v in g32.reshape(3, -1).T:
        ss = (ss + (v * v).reshape(3, 1, 1)).astype(np.float32)
    nrm = _bf16(np.sqrt(ss))
    t = _bf16(nrm * np.float32(1.02))
    den = _bf16(t + np.float32(1e-6))
    x32 = _bf16(g32 / den.astype(np.float32))
    assert np.all(np.abs(x32 - x) <= rad)
    # ||G|| = 5 exactly (a 3-4 right triangle): den = bf16(bf16(5.1) + 1e-6)
    g2 = np.zeros((1, 8, 8))
    g2[0, 0, 0], g2[0, 1, 1] = 3.0, 4.0
    x2, _ = pe.normalize_rounded(g2)
    den2 = _bf16(_bf16(5.0 * np.float64(np.float32(1.02))) + np.float64(np.float32(1e-6)))
    assert x2[0, 0, 0] == _bf16(3.0 / den2) and x2[0, 1, 1] == _bf16(4.0 / den2)


def _rounded_chain(g, steps=5):
    x, _ = pe.normalize_rounded(g)
    tall = x.shape[-2] > x.shape[-1]
    for a, b, c in pe.POLAR_EXPRESS_COEFFS[:steps]:
        xt = np.swapaxes(x, -1, -2)
        A, _ = pe.gemm_rounded(xt, x) if tall else pe.gemm_rounded(x, xt)
        B, _ = pe.gemm_rounded(A, A, c, b, A)
        x, _ = pe.gemm_rounded(x, B, 1.0, a, x) if tall else pe.gemm_rounded(B, x, 1.0, a, x)
    return x


@pytest.mark.parametrize("m,n", [(32, 48), (48, 32)])
def test_rounded_chain_stays_close_to_the_float64_iteration(m, n):
    """The bf16-rounding-point chain (what a bf16 evaluation computes) against the float64 iteration on the
    same bf16 input: the same polynomials on the singular values, perturbed by one bf16 rounding per
    product; after five steps the Frobenius distance stays within 5 % and the singular values within the
    band the float64 iteration produces."""
    g = _bf16(np.random.default_rng(m).standard_normal((1, m, n)))
    ref = pe.polar_express(g)
    got = _rounded_chain(g)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 5e-2, rel
    sv_ref = np.linalg.svd(ref[0], compute_uv=False)
    sv = np.linalg.svd(got[0], compute_uv=False)
    assert abs(sv.max() - sv_ref.max()) < 0.1 and abs(sv.min() - sv_ref.min()) < 0.1
