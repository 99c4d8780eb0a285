"""Pure-Python brute force of the attention forward for tiny inputs (T <= 8).

TEST INFRASTRUCTURE. A second, independently written evaluation of the same definition as
attn_oracle.c, used to pin it. It deliberately uses other formulations of each step:

* RoPE as complex multiplication: pair i is z = x[i] + 1j*x[i + D/2] and the rotated pair is
  z * exp(-1j * t * base^(-2i/D)); real and imaginary parts give y1 = x1 cos + x2 sin and
  y2 = -x1 sin + x2 cos (habr "Autoresearch" deep dive, train.py listing, apply_rotary_emb).
* The mask as FlashAttention's (left, right) window around the diagonal: left = W (unbounded
  if W < 0), right = 0 when causal, else W (unbounded if W < 0); key j is visible to query i
  iff i - left <= j <= i + right (listing, flash_attn_func(..., causal=True,
  window_size=(W, 0)); "geometry_of_andrea" page, "A Máscara Causal").
* bf16 rounding via math.frexp and Python's round-half-even on the scaled mantissa.
* Sums with math.fsum.
"""
from __future__ import annotations

import cmath
import math
from typing import List, Sequence, Tuple

Mat = List[List[float]]


def round_bf16(x: float) -> float:
    """Nearest bf16 value (8 significant bits), ties to even."""
    if x == 0.0 or math.isinf(x) or math.isnan(x):
        return x
    m, e = math.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    if e - 8 < -133:
        return round(x * 2.0 ** 133) / 2.0 ** 133
    return math.ldexp(round(m * 256.0), e - 8)


def rope(x: Sequence[float], t: int, base: float) -> List[float]:
    D = len(x)
    half = D // 2
    y = [0.0] * D
    for i in range(half):
        z = complex(x[i], x[i + half]) * cmath.exp(-1j * t * base ** (-2.0 * i / D))
        y[i], y[i + half] = z.real, z.imag
    return y


def rmsnorm(x: Sequence[float], eps: float) -> List[float]:
    ms = math.fsum(a * a for a in x) / len(x)
    return [a / math.sqrt(ms + eps) for a in x]


def visible(i: int, j: int, window: int, causal: bool) -> bool:
    left = math.inf if window < 0 else window
    right = 0 if causal else (math.inf if window < 0 else window)
    return i - left <= j <= i + right


def head_forward(q: Mat, k: Mat, v: Mat, window: int, causal: bool, rope_base: float, eps: float,
                 round_qk: bool = True) -> Tuple[Mat, List[float], Mat]:
    """One head: q, k, v are T x D lists of floats (already bf16 values).
    Returns (out T x D, lse[T], weights T x T)."""
    T, D = len(q), len(q[0])

    def prep(x, t):
        y = list(x)
        if rope_base > 0:
            y = rope(y, t, rope_base)
        if eps >= 0:
            y = rmsnorm(y, eps)
        if round_qk:
            y = [round_bf16(a) for a in y]
        return y

    qh = [prep(q[t], t) for t in range(T)]
    kh = [prep(k[t], t) for t in range(T)]
    out, lse, P = [], [], []
    for i in range(T):
        scores = {}
        for j in range(T):
            if visible(i, j, window, causal):
                scores[j] = math.fsum(a * b for a, b in zip(qh[i], kh[j])) / math.sqrt(D)
        m = max(scores.values())
        z = math.fsum(math.exp(s - m) for s in scores.values())
        w = [math.exp(scores[j] - m) / z if j in scores else 0.0 for j in range(T)]
        out.append([math.fsum(w[j] * v[j][d] for j in range(T)) for d in range(D)])
        lse.append(m + math.log(z))
        P.append(w)
    return out, lse, P


def forward(q4, k4, v4, window: int, causal: bool, rope_base: float, eps: float, round_qk: bool = True):
    """q4, k4, v4: nested lists or float arrays indexed [b][t][h][d].
    Returns (out [b][t][h][d], lse [b][h][t])."""
    B, T, H = len(q4), len(q4[0]), len(q4[0][0])
    out = [[[None] * H for _ in range(T)] for _ in range(B)]
    lse = [[[0.0] * T for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            qq = [[float(x) for x in q4[b][t][h]] for t in range(T)]
            kk = [[float(x) for x in k4[b][t][h]] for t in range(T)]
            vv = [[float(x) for x in v4[b][t][h]] for t in range(T)]
            o, l, _ = head_forward(qq, kk, vv, window, causal, rope_base, eps, round_qk)
            for t in range(T):
                out[b][t][h] = o[t]
                lse[b][h][t] = l[t]
    return out, lse
