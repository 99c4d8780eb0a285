"""Oracle for the Polar Express orthogonalisation of the Muon optimiser step (NEXT-4), float64.

TEST INFRASTRUCTURE ONLY, like the rest of this package.

What it computes (habr "Autoresearch" deep dive, train.py listing, optimiser section: the Muon step
orthogonalises the momentum-mixed gradient with `polar_express_coeffs`), per matrix G of a batch:
    X = G / (||G||_F * 1.02 + 1e-6)
    for each of the first `steps` coefficient triples (a, b, c):
        tall (rows > cols):  A = X^T X,  X = a X + X (b A + c A^2)
        otherwise:           A = X X^T,  X = a X + (b A + c A^2) X
Each step maps every singular value s of X to a s + b s^3 + c s^5 and keeps the singular vectors,
so the result approximates the polar factor U V^T of G. The listing runs this in bf16; the oracle
evaluates the same steps in float64.

The five coefficient triples are the listing's table, kept as data (they define the method).

Pinned by tests/test_oracle_polar.py: the iteration equals the polynomial applied to the singular
values from numpy's SVD, the wide form on G^T equals the transpose of the tall form on G, and for
well-conditioned G the result is close to U V^T. The rounding-point functions below (gemm_rounded,
normalize_rounded) are pinned by exact integer cases, by float32 evaluations landing inside their radii,
and by the rounded chain staying close to the float64 iteration.
"""
from __future__ import annotations

import numpy as np

# (a, b, c) per step, in the listing's order
POLAR_EXPRESS_COEFFS = (
    (8.156554524902461, -22.48329292557795, 15.878769915207462),
    (4.042929935166739, -2.808917465908714, 0.5000178451051316),
    (3.8916678022926607, -2.772484153217685, 0.5060648178503393),
    (3.285753657755655, -2.3681294933425376, 0.46449024233003106),
    (2.3465413258596377, -1.7097828382687081, 0.42323551169305323),
)


def polar_express(g, steps: int = 5) -> np.ndarray:
    """g: [..., m, n] (any real dtype or a torch tensor); returns float64 [..., m, n]."""
    if not isinstance(g, np.ndarray):
        g = g.detach().cpu().double().numpy()
    x = np.asarray(g, dtype=np.float64)
    fro = np.sqrt(np.sum(x * x, axis=(-2, -1), keepdims=True))
    x = x / (fro * 1.02 + 1e-6)
    tall = x.shape[-2] > x.shape[-1]
    for a, b, c in POLAR_EXPRESS_COEFFS[:steps]:
        if tall:
            A = np.swapaxes(x, -1, -2) @ x
            x = a * x + x @ (b * A + c * (A @ A))
        else:
            A = x @ np.swapaxes(x, -1, -2)
            x = a * x + (b * A + c * (A @ A)) @ x
    return x


# ---------------------------------------------------------------------------------------------
# The same steps at bf16 rounding points, one operation at a time (for checking a bf16 GPU
# evaluation step by step). Every result is the exact value rounded once to bf16; each carries an
# ambiguity radius: the largest distance to the bf16 value any single-precision evaluation within
# the stated budget can round to.


def _as_f64(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _round_with_radius(exact: np.ndarray, budget: np.ndarray):
    from . import round_bf16_array

    y = round_bf16_array(exact)
    lo, hi = round_bf16_array(exact - budget), round_bf16_array(exact + budget)
    return y, np.maximum(np.abs(hi - y), np.abs(y - lo))


def gemm_rounded(p, q, alpha: float = 1.0, beta: float = 0.0, r=None):
    """D = bf16(alpha * P Q + beta * R) for batched P [.., M, K], Q [.., K, N] (bf16 values), with the
    radius of a single-precision evaluation: the K products accumulated in fp32 in any order with any
    rounding of the partial sums (at most 2 K 2^-24 sum |P| |Q|, twice the round-to-nearest bound), then
    alpha times that plus beta R in fp32 (2 * 2^-24 of |alpha P Q| + |beta R|). alpha and beta are
    taken as the fp32 values they are passed as."""
    pp, qq = _as_f64(p), _as_f64(q)
    a = float(np.float32(alpha))
    b = float(np.float32(beta))
    prod = pp @ qq
    mag = np.abs(pp) @ np.abs(qq)
    K = pp.shape[-1]
    rr = _as_f64(r) if r is not None else np.zeros_like(prod)
    exact = a * prod + b * rr
    budget = abs(a) * 2.0 * K * 2.0 ** -24 * mag + 2.0 * 2.0 ** -24 * (np.abs(a * prod) + np.abs(b * rr))
    return _round_with_radius(exact, budget)


def normalize_rounded(g):
    """X = G / (||G||_F * 1.02 + 1e-6) at the listing's bf16 rounding points, per matrix of [.., m, n]:
    nrm = bf16(||G||_F), t = bf16(nrm * fp32(1.02)), den = bf16(t + fp32(1e-6)), X = bf16(G / den).
    Radius: the sum of squares accumulated in fp32 in any order (relative 2 mn 2^-24), its square root
    correctly rounded (2^-24 more), every later value within one fp32 rounding of its exact form; each
    candidate chain of bf16 values is followed to the end and the radius is the largest distance from
    the exact-then-rounded X."""
    from . import round_bf16_array

    gg = _as_f64(g)
    ss = np.sum(gg * gg, axis=(-2, -1), keepdims=True)
    mn = gg.shape[-2] * gg.shape[-1]
    f102 = float(np.float32(1.02))
    f1e6 = float(np.float32(1e-6))

    def chain(rel, e1, e2, e3):
        nrm = round_bf16_array(np.sqrt(ss * (1.0 + rel)))
        t = round_bf16_array(nrm * f102 * (1.0 + e1 * 2.0 ** -23))
        den = round_bf16_array((t + f1e6) * (1.0 + e2 * 2.0 ** -23))
        return round_bf16_array(gg / den * (1.0 + e3 * 2.0 ** -23))

    base = chain(0.0, 0, 0, 0)
    radius = np.zeros_like(gg)
    d = (2.0 * mn + 2.0) * 2.0 ** -24
    for rel in (-d, 0.0, d):
        for e1 in (-1, 0, 1):
            for e2 in (-1, 0, 1):
                for e3 in (-1, 0, 1):
                    radius = np.maximum(radius, np.abs(chain(rel, e1, e2, e3) - base))
    return base, radius
