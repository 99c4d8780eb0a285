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
well-conditioned G the result is close to U V^T.
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
