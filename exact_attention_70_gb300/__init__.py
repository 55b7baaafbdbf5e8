"""Exact tiled scaled-dot-product attention for GB300 (sm_103a).

The compute lives in ``libattn.so`` (hand-written CUDA behind a C ABI declared in
``include/attn.h``); this package only marshals arguments.  ``attn_fwd`` and
``attn_decode_kvcache`` are loaded on first use and raise if the library is missing.
"""

__all__ = ["attn_fwd", "attn_decode_kvcache", "attn_fwd_workspace_bytes",
           "attn_decode_workspace_bytes", "attn_get_device_status", "AttnError"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
