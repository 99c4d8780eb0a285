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


def call_bwd(b, **kw):
    a = dict(q=FAKE, k=FAKE + (1 << 24), v=FAKE + (2 << 24), out=FAKE + (3 << 24), lse=FAKE + (4 << 24),
             dout=FAKE + (5 << 24), dq=FAKE + (6 << 24), dk=FAKE + (7 << 24), dv=FAKE + (8 << 24),
             ws=FAKE + (9 << 24), ws_bytes=None, B=1, H=2, H_kv=2, T=64, D=64, window=-1, causal=1,
             rope_base=10000.0, eps=1e-6)
    a.update(kw)
    if a["ws_bytes"] is None:
        a["ws_bytes"] = b.attn_bwd_workspace_bytes(a["B"], a["H"], a["H_kv"], a["T"], a["D"])
    return b.lib.attn_bwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["dout"], a["dq"], a["dk"], a["dv"], a["ws"],
                          a["ws_bytes"], a["B"], a["H"], a["H_kv"], a["T"], a["D"], a["window"], a["causal"],
                          a["rope_base"], a["eps"], None)


def test_bwd_workspace_size(binding):
    B, H, Hkv, T, D = 2, 4, 2, 300, 64
    n = binding.attn_bwd_workspace_bytes(B, H, Hkv, T, D)
    # q^ and k^ in bf16; delta and -lse log2(e) in fp32 rows of whole 128-query tiles; the dq^
    # accumulator in fp32; a work counter; each part padded to 256 bytes
    Tp = (T + 127) // 128 * 128
    parts = [B * T * H * D * 2, B * T * Hkv * D * 2, B * H * Tp * 4, B * H * Tp * 4, B * T * H * D * 4, 4]
    assert sum(parts) <= n <= sum(parts) + 6 * 256
    assert n % 256 == 0
    assert binding.attn_bwd_workspace_bytes(0, H, Hkv, T, D) == 0
    assert binding.attn_bwd_workspace_bytes(B, H, Hkv, -1, D) == 0


def test_bwd_host_validation_codes(binding):
    E = binding
    for name in ("q", "k", "v", "out", "lse", "dout", "dq", "dk", "dv", "ws"):
        assert call_bwd(binding, **{name: 0}) == E.ATTN_ERR_INVALID_ARG, name
    assert call_bwd(binding, dq=FAKE + (6 << 24) + 8) == E.ATTN_ERR_INVALID_ARG  # misaligned
    assert call_bwd(binding, ws=FAKE + (9 << 24) + 16) == E.ATTN_ERR_INVALID_ARG  # workspace not 256-aligned
    assert call_bwd(binding, ws_bytes=1024) == E.ATTN_ERR_INVALID_ARG  # workspace too small
    assert call_bwd(binding, H_kv=3) == E.ATTN_ERR_INVALID_ARG
    assert call_bwd(binding, causal=2) == E.ATTN_ERR_INVALID_ARG
    assert call_bwd(binding, eps=float("inf")) == E.ATTN_ERR_INVALID_ARG
    assert call_bwd(binding, dq=FAKE + 4096) == E.ATTN_ERR_INVALID_ARG  # dq overlaps q
    assert call_bwd(binding, dv=FAKE + (9 << 24) + 256) == E.ATTN_ERR_INVALID_ARG  # dv overlaps the workspace
    assert call_bwd(binding, dk=FAKE + (6 << 24) + 1024) == E.ATTN_ERR_INVALID_ARG  # dk overlaps dq
    assert call_bwd(binding, D=48) == E.ATTN_ERR_UNSUPPORTED
    assert call_bwd(binding) == E.ATTN_ERR_NOT_INITIALIZED
    assert call_bwd(binding, H=4, H_kv=1, D=128, T=300, window=100) == E.ATTN_ERR_NOT_INITIALIZED


def test_value_gate_host_validation_codes(binding):
    E = binding
    lib = binding.lib
    q, k, v, ve = FAKE, FAKE + (1 << 24), FAKE + (2 << 24), FAKE + (3 << 24)
    x, w, out, lse = FAKE + (4 << 24), FAKE + (5 << 24), FAKE + (6 << 24), FAKE + (7 << 24)
    ws = FAKE + (8 << 24)
    assert binding.attn_fwd_ve_workspace_bytes(1, 2, 64) == 512  # 1 * 64 * 2 fp32 factors
    assert binding.attn_fwd_ve_workspace_bytes(0, 2, 64) == 0

    def call(**kw):
        a = dict(q=q, k=k, v=v, ve=ve, x=x, xs=64, w=w, out=out, lse=lse, ws=ws, wsb=512, B=1, H=4, Hkv=2, T=64, D=64)
        a.update(kw)
        return lib.attn_fwd_ve(a["q"], a["k"], a["v"], a["ve"], a["x"], a["xs"], a["w"], a["out"], a["lse"], a["ws"],
                               a["wsb"], a["B"], a["H"], a["Hkv"], a["T"], a["D"], -1, 1, 10000.0, 1e-6, None)

    assert call(ve=0) == E.ATTN_ERR_INVALID_ARG
    assert call(x=0) == E.ATTN_ERR_INVALID_ARG
    assert call(w=0) == E.ATTN_ERR_INVALID_ARG
    assert call(ve=ve + 8) == E.ATTN_ERR_INVALID_ARG   # misaligned
    assert call(xs=16) == E.ATTN_ERR_INVALID_ARG       # fewer than 32 channels per row
    assert call(xs=36) == E.ATTN_ERR_INVALID_ARG       # rows not 16-byte aligned
    assert call(out=ve + 256) == E.ATTN_ERR_INVALID_ARG  # out overlaps ve
    assert call(ws=0) == E.ATTN_ERR_INVALID_ARG
    assert call(wsb=256) == E.ATTN_ERR_INVALID_ARG     # workspace too small
    assert call(ws=out + 64) == E.ATTN_ERR_INVALID_ARG  # workspace overlaps out
    assert call(D=48) == E.ATTN_ERR_UNSUPPORTED
    assert call() == E.ATTN_ERR_NOT_INITIALIZED
    assert call(xs=32) == E.ATTN_ERR_NOT_INITIALIZED


def test_polar_header_and_exports(binding):
    """include/polar.h declares exactly the pe_* / polar_express symbols the library exports."""
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "polar.h")).read(), flags=re.S)
    declared = set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:pe_|polar_)\w+)\s*\(", text, flags=re.M))
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T ((?:pe_|polar_)\w+)", out))
    assert declared == exported == {"pe_workspace_bytes", "pe_step_flops", "pe_normalize", "pe_step", "polar_express"}
    from sliding_window_attention_04_b300 import polar

    assert set(polar.EXPORTED) == exported


def test_polar_host_validation_codes(binding):
    from sliding_window_attention_04_b300 import polar

    E, lib = binding, binding.lib
    x, y, ws = FAKE, FAKE + (1 << 24), FAKE + (2 << 24)
    nb = polar.workspace_bytes(2, 64, 96)
    assert nb >= 2 * 64 * 64 * 2 * 2 + 2 * 64 * 96 * 2 and nb % 256 == 0
    assert polar.workspace_bytes(0, 64, 96) == 0
    assert polar.step_flops(2, 64, 96) == 0.0  # not initialised
    assert lib.pe_step(x, y, 2, 64, 96, 0, ws, nb, None) == E.ATTN_ERR_NOT_INITIALIZED
    assert lib.pe_step(x, y, 2, 64, 100, 0, ws, nb, None) == E.ATTN_ERR_INVALID_ARG   # n not a multiple of 8
    assert lib.pe_step(x, y, 2, 64, 96, 5, ws, nb, None) == E.ATTN_ERR_INVALID_ARG    # no sixth triple
    assert lib.pe_step(x, y, 2, 64, 96, 0, ws, nb - 256, None) == E.ATTN_ERR_INVALID_ARG
    assert lib.pe_step(x, x + 64, 2, 64, 96, 0, ws, nb, None) == E.ATTN_ERR_INVALID_ARG  # X and Y overlap
    assert lib.pe_step(x, y, 2, 64, 96, 0, ws + 16, nb, None) == E.ATTN_ERR_INVALID_ARG  # workspace alignment
    assert lib.polar_express(x, y, 2, 64, 96, 6, ws, nb, None) == E.ATTN_ERR_INVALID_ARG
    assert lib.polar_express(x, y, 2, 64, 96, 5, ws, nb, None) == E.ATTN_ERR_NOT_INITIALIZED
    assert lib.pe_normalize(x, y, 0, 64, 96, ws, nb, None) == E.ATTN_ERR_INVALID_ARG
    assert lib.pe_normalize(x, y, 2, 64, 96, ws, nb - 256, None) == E.ATTN_ERR_INVALID_ARG  # no room for the partials
    assert lib.pe_normalize(x, x + 64, 2, 64, 96, ws, nb, None) == E.ATTN_ERR_INVALID_ARG  # partial overlap
    assert lib.pe_normalize(x, x, 2, 64, 96, ws, nb, None) == E.ATTN_ERR_NOT_INITIALIZED   # in place is allowed
    # the partial sums: at most 1024 per matrix, 16384 elements per chunk for small matrices
    big = polar.workspace_bytes(1, 4096, 8192)
    assert big >= 2 * 4096 * 4096 * 2 + 4096 * 8192 * 2 + 1024 * 4
