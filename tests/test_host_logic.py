"""Host-side logic that needs no GPU: the SSSL window schedule, the FLOP count, the inputs."""
import numpy as np
import torch

from sliding_window_attention_04_b300 import configs
from sliding_window_attention_04_b300.inputs import layer_seed, make_qkv


def test_window_schedule_sssl():
    # habr "Autoresearch" deep dive, train.py listing, _compute_window_sizes: S = T // 2,
    # L = T, pattern cycled over layers, last layer forced to L.
    assert configs.window_schedule("SSSL", 4, 1024) == [512, 512, 512, 1024]
    assert configs.window_schedule("SSSL", 12, 1024) == [512, 512, 512, 1024] * 3
    assert configs.window_schedule("SSSL", 16, 1024) == [512, 512, 512, 1024] * 4
    # depth 8 example of the Korean deep dive: layers 0-2 S, 3 L, 4-6 S, 7 L
    assert configs.window_schedule("SSSL", 8, 2048) == [1024] * 3 + [2048] + [1024] * 3 + [2048]
    # last layer is forced to L even when the pattern would give S there
    assert configs.window_schedule("SSSL", 6, 1024) == [512, 512, 512, 1024, 512, 1024]
    assert configs.window_schedule("S", 3, 100) == [50, 50, 100]
    assert configs.window_schedule("sssl", 1, 10) == [10]


def test_window_schedule_rejects_bad_pattern():
    import pytest

    with pytest.raises(ValueError):
        configs.window_schedule("SXL", 4, 1024)
    with pytest.raises(ValueError):
        configs.window_schedule("", 4, 1024)


def test_flop_count_matches_enumeration():
    for T in (1, 5, 64, 130):
        for window in (-1, 0, 1, 7, T // 2, T, 3 * T):
            for causal in (True, False):
                brute = sum(configs.n_allowed_keys(i, T, window, causal) for i in range(T))
                assert configs.n_unmasked(T, window, causal) == brute


def test_workload_totals():
    w = configs.workloads()[2]
    assert (w.B, w.H, w.T, w.D, len(w.layers)) == (32, 12, 1024, 64, 12)
    assert [l.window for l in w.layers] == [512, 512, 512, 1024] * 3
    assert abs(w.flops() / 1e9 - 503.34) < 0.01
    assert abs(w.bytes() / 1e6 - 2434.79) < 0.01


def test_inputs_are_seeded_bf16():
    a = make_qkv(2, 8, 3, 16, seed=layer_seed(2, 5))
    b = make_qkv(2, 8, 3, 16, seed=2005)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and x.shape == (2, 8, 3, 16)
        assert torch.equal(x, y)
    c = make_qkv(2, 8, 3, 16, seed=2006)
    assert not torch.equal(a[0], c[0])
    assert abs(float(a[2].float().std()) - 1.0) < 0.2
    assert np.isfinite(a[0].float().numpy()).all()
