"""Paged-KV attention with a learned relative-position bias for sm_103a GPUs.

The compute lives in libinkling_rel_attn.so (C ABI, include/inkling_rel_attn.h);
this package is its thin Python binding.  Importing the package does not load
the library; the first call does, and fails loudly if it was not built.
"""

from .ops import (  # noqa: F401
    InklingError,
    choose_splits,
    decode,
    decode_inputs,
    decode_multi,
    decode_multi_workspace_bytes,
    decode_workspace_bytes,
    kv_append,
    kv_conv_append,
    prefill,
    prefill_inputs,
)

__all__ = ["InklingError", "choose_splits", "decode", "decode_inputs", "decode_multi",
           "decode_multi_workspace_bytes", "decode_workspace_bytes",
           "kv_append", "kv_conv_append", "prefill", "prefill_inputs"]
