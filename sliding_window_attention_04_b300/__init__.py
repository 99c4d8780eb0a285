"""B300 (sm_103a) attention forward: QK-RMSNorm + RoPE + causal / sliding-window softmax(QK^T/sqrt(D))V.

The computation lives in the CUDA library `_lib/libswa_attn.so` (C ABI: include/attn.h); the
binding `sliding_window_attention_04_b300.attn` exposes the same names to Python. Importing the
package itself does not load the library, so the input generator and the workload tables can be
used on machines without a GPU; the first access to a binding name loads it, and raises if the
library is missing.
"""
_BINDING_NAMES = ("attn_init", "attn_fwd", "attn_destroy", "attn_device_status", "status_string", "AttnError")


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import attn as _attn

        return getattr(_attn, name)
    raise AttributeError(name)


__all__ = list(_BINDING_NAMES)
