"""The C-ABI library loads, exports every function include/attn.h declares, and rejects bad
arguments on the host before touching the GPU (runs on machines without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def binding():
    from sliding_window_attention_04_b300.csrc import build

    build.build()
    from sliding_window_attention_04_b300 import attn

    return attn


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_init", "attn_fwd", "attn_destroy", "attn_status_string", "attn_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (attn_\w+)", out))
    assert set(declared_functions()) == exported
    assert set(binding.EXPORTED) == exported


def test_status_strings(binding):
    assert binding.status_string(0) == "ATTN_OK"
    assert binding.status_string(-2) == "ATTN_ERR_INVALID_ARG"
    assert binding.status_string(-5) == "ATTN_ERR_DEVICE_TIMEOUT"
    assert binding.status_string(-7) == "ATTN_ERR_SCRATCH_LIMIT"
    assert binding.status_string(12345) == "ATTN_ERR_UNKNOWN"


FAKE = 1 << 20  # a 16-byte-aligned address that is never dereferenced by these calls


def call(b, **kw):
    a = dict(q=FAKE, k=FAKE + (1 << 24), v=FAKE + (2 << 24), out=FAKE + (3 << 24), lse=FAKE + (4 << 24), B=1, H=2,
             T=64, D=64, window=-1, causal=1, rope_base=10000.0, eps=1e-6, stream=None)
    a.update(kw)
    return b.attn_fwd_raw(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["H"], a["T"], a["D"], a["window"],
                          a["causal"], a["rope_base"], a["eps"], a["stream"])


def test_host_validation_codes(binding):
    E = binding
    assert call(binding, q=0) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, out=0) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, v=FAKE + 8) == E.ATTN_ERR_INVALID_ARG  # misaligned
    assert call(binding, lse=FAKE + (4 << 24) + 2) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, B=0) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, H=-1) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, T=0) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, causal=2) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, rope_base=-1.0) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, rope_base=float("inf")) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, eps=float("nan")) == E.ATTN_ERR_INVALID_ARG
    assert call(binding, B=1 << 15, T=1 << 10, H=32, D=64) == E.ATTN_ERR_INVALID_ARG  # >= 2^31 elements
    assert call(binding, out=FAKE + 64) == E.ATTN_ERR_INVALID_ARG  # out overlaps q
    assert call(binding, lse=FAKE + (3 << 24) + 16) == E.ATTN_ERR_INVALID_ARG  # lse overlaps out
    assert call(binding, D=48) == E.ATTN_ERR_UNSUPPORTED
    assert call(binding, D=256) == E.ATTN_ERR_UNSUPPORTED
    # a valid request on a library that has not been initialised
    assert call(binding) == E.ATTN_ERR_NOT_INITIALIZED
    assert call(binding, lse=None) == E.ATTN_ERR_NOT_INITIALIZED
    assert binding.attn_device_status() == E.ATTN_ERR_NOT_INITIALIZED


def call_gqa(b, **kw):
    a = dict(q=FAKE, k=FAKE + (1 << 24), v=FAKE + (2 << 24), out=FAKE + (3 << 24), lse=FAKE + (4 << 24), B=1, H=4,
             H_kv=2, T=64, D=64, window=-1, causal=1, rope_base=10000.0, eps=1e-6, stream=None)
    a.update(kw)
    return b.attn_fwd_gqa_raw(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["H"], a["H_kv"], a["T"], a["D"],
                              a["window"], a["causal"], a["rope_base"], a["eps"], a["stream"])


def test_gqa_host_validation_codes(binding):
    E = binding
    for bad in (0, -1, 3, 8):  # not a divisor of H = 4, or more K/V heads than query heads
        assert call_gqa(binding, H_kv=bad) == E.ATTN_ERR_INVALID_ARG, bad
    assert call_gqa(binding, k=FAKE + 8) == E.ATTN_ERR_INVALID_ARG  # misaligned
    # out [1, 64, 4, 64] bf16 = 32 KB; k [1, 64, 2, 64] = 16 KB: out placed 8 KB into k overlaps it
    assert call_gqa(binding, out=FAKE + (1 << 24) + 8192) == E.ATTN_ERR_INVALID_ARG
    # ... and right after the end of k does not
    assert call_gqa(binding, out=FAKE + (1 << 24) + 16384) == E.ATTN_ERR_NOT_INITIALIZED
    assert call_gqa(binding) == E.ATTN_ERR_NOT_INITIALIZED
    assert call_gqa(binding, H_kv=4) == E.ATTN_ERR_NOT_INITIALIZED
    assert call_gqa(binding, H_kv=1, D=128) == E.ATTN_ERR_NOT_INITIALIZED


def test_init_without_device(binding):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert binding.lib.attn_init(0) == binding.ATTN_ERR_NO_DEVICE
    binding.attn_destroy()  # idempotent, nothing to free
    binding.attn_destroy()


def test_binding_rejects_cpu_tensors(binding):
    import torch

    x = torch.zeros((1, 4, 1, 32), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.attn_fwd(x, x, x)
