"""Workload shapes, the SSSL window schedule and the unmasked-FLOP count used by the benchmark.

Shapes follow the ANDREA family table ("grow_a_language_model_intro" page, section "Uma Família
de Três": d_model / heads / T = 1024, so D = d_model / heads). The per-layer window schedule
follows `GPT._compute_window_sizes` in the train.py listing of the habr "Autoresearch" deep dive:
the pattern string is cycled over the layers, 'S' is a window of `seq_len // 2`, 'L' is
`seq_len` (full causal), and the last layer is always forced to 'L'. The window value is handed
to the attention call unchanged as `window_size=(W, 0)` (CausalSelfAttention.forward), i.e. a
query at position i sees keys j with i - W <= j <= i.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Tuple


def window_schedule(pattern: str, n_layer: int, seq_len: int) -> List[int]:
    """Per-layer window W for a pattern such as "SSSL" (last layer forced to full context)."""
    pattern = pattern.upper()
    if not pattern or any(c not in "SL" for c in pattern):
        raise ValueError(f"pattern must be a non-empty string over 'S'/'L': {pattern!r}")
    if n_layer < 1:
        raise ValueError("n_layer must be >= 1")
    long_w = seq_len
    short_w = seq_len // 2
    sizes = [long_w if pattern[i % len(pattern)] == "L" else short_w for i in range(n_layer)]
    sizes[-1] = long_w
    return sizes


def n_allowed_keys(i: int, T: int, window: int, causal: bool) -> int:
    """|J(i)|: how many keys j in [0, T) query i may attend to (FA window convention)."""
    lo = 0 if window < 0 else max(0, i - window)
    if causal:
        hi = i
    elif window < 0:
        hi = T - 1
    else:
        hi = min(T - 1, i + window)
    return max(0, hi - lo + 1)


def n_unmasked(T: int, window: int, causal: bool = True) -> int:
    """Number of unmasked score entries of one (b, h) pair: sum over i of |J(i)|.

    Closed form for the causal case: T(T+1)/2 when window < 0 or window >= T - 1, else
    W(W+1)/2 + (T - W)(W + 1) with W = window. The non-causal case is summed directly.
    """
    if causal:
        if window < 0 or window >= T - 1:
            return T * (T + 1) // 2
        W = window
        return W * (W + 1) // 2 + (T - W) * (W + 1)
    return sum(n_allowed_keys(i, T, window, causal) for i in range(T))


def attn_flops(B: int, H: int, T: int, D: int, window: int, causal: bool = True) -> int:
    """Algorithmic FLOPs of one forward call: 2*D for q.k plus 2*D for p*v per unmasked entry."""
    return 4 * D * n_unmasked(T, window, causal) * B * H


def attn_bytes(B: int, H: int, T: int, D: int, with_lse: bool = True) -> int:
    """Compulsory HBM bytes of one call: read q, k, v and write out (bf16), plus the fp32 LSE."""
    return 2 * B * T * H * D * 4 + (4 * B * H * T if with_lse else 0)


@dataclass(frozen=True)
class Layer:
    window: int
    causal: bool = True


@dataclass(frozen=True)
class Workload:
    """One named workload: a shape and its list of layers (each layer gets its own inputs)."""

    name: str
    index: int
    B: int
    H: int
    T: int
    D: int
    layers: Tuple[Layer, ...] = field(default_factory=tuple)
    rope_base: float = 10000.0
    eps: float = 1e-6

    def flops(self) -> int:
        return sum(attn_flops(self.B, self.H, self.T, self.D, l.window, l.causal) for l in self.layers)

    def bytes(self) -> int:
        return len(self.layers) * attn_bytes(self.B, self.H, self.T, self.D)


def _sssl(n_layer: int, T: int) -> Tuple[Layer, ...]:
    return tuple(Layer(w, True) for w in window_schedule("SSSL", n_layer, T))


def workloads() -> List[Workload]:
    """The five workloads: tiny full-causal, ANDREA-12M/120M/480M-shaped SSSL stacks, and the
    sequence-length sweep (one S and one L layer per T, B = 32768 / T)."""
    w = [
        Workload("tiny full-causal B1 H12 T256 D32", 0, 1, 12, 256, 32, (Layer(256, True),)),
        Workload("ANDREA-12M shape SSSL B16 H12 T1024 D32", 1, 16, 12, 1024, 32, _sssl(4, 1024)),
        Workload("ANDREA-120M shape SSSLx3 B32 H12 T1024 D64", 2, 32, 12, 1024, 64, _sssl(12, 1024)),
        Workload("ANDREA-480M shape SSSLx4 B16 H24 T1024 D64", 3, 16, 24, 1024, 64, _sssl(16, 1024)),
    ]
    return w


def sweep_workloads() -> List[Workload]:
    """Sequence-length sweep: H=12, D=64, T in {1024..8192}, B = 32768/T, one S(T/2) + one L layer."""
    out = []
    for T in (1024, 2048, 4096, 8192):
        out.append(Workload(f"sweep T{T} B{32768 // T} H12 D64", 4, 32768 // T, 12, T, 64,
                            (Layer(T // 2, True), Layer(T, True))))
    return out


def extra_workloads() -> List[Workload]:
    """Shapes beyond the five workloads, for extra measurements: the autoresearch default attention
    shape (habr "Autoresearch" deep dive, train.py listing: sequence_len 2048, head_dim 128; 4 heads
    per layer at the default depth, B = 128), one S layer (W = T/2) and one L layer."""
    return [Workload("autoresearch default shape B128 H4 T2048 D128", 5, 128, 4, 2048, 128,
                     (Layer(1024, True), Layer(2048, True)))]


def by_name(prefix: str) -> Workload:
    for w in workloads() + sweep_workloads() + extra_workloads():
        if w.name.startswith(prefix):
            return w
    raise KeyError(prefix)
