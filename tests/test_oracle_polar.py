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
