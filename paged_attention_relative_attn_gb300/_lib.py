"""ctypes binding of libinkling_rel_attn.so: argument marshalling only.

Every function here has the name and the argument order of the C entry point
declared in include/inkling_rel_attn.h; pointers are passed as Python ints
(device addresses), the stream as its integer handle.  Loading fails loudly
when the library has not been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libinkling_rel_attn.so")

#: C entry points (the names declared in include/inkling_rel_attn.h)
EXPORTED = (
    "inkling_rel_attn_decode",
    "inkling_rel_attn_decode_noalloc",
    "inkling_rel_attn_decode_multi",
    "inkling_rel_attn_decode_multi_workspace_size",
    "inkling_rel_attn_prefill",
    "inkling_rel_attn_kv_append",
    "inkling_rel_attn_kv_conv_append",
    "inkling_rel_attn_choose_splits",
    "inkling_rel_attn_decode_workspace_size",
    "inkling_rel_attn_prefill_workspace_size",
    "inkling_rel_attn_selftest_timeout",
    "inkling_rel_attn_error_string",
    "inkling_rel_attn_version",
)

_lib = None

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_f32 = ctypes.c_float

_SIGS = {
    "inkling_rel_attn_decode": (ctypes.c_int, [
        _p, _p, _p, _p, _i32, _p, _p,               # q k v page_table stride seq_lens rel
        _i32, _i32, _i32, _i32, _i32, _i32, _i32,   # B H_q H_kv D page_size num_pages R
        _i32, _f32, _i32,                           # window scale max_seq_len
        _p, _p, _p, _sz, _i32, _p, _p]),            # out lse ws ws_bytes splits err stream
    "inkling_rel_attn_decode_noalloc": (ctypes.c_int, [
        _p, _p, _p, _p, _i32, _p, _p,               # q k v page_table stride seq_lens rel
        _i32, _i32, _i32, _i32, _i32, _i32, _i32,   # B H_q H_kv D page_size num_pages R
        _i32, _f32, _i32,                           # window scale max_seq_len
        _p, _p, _i32, _p, _p]),                     # out lse splits err stream
    "inkling_rel_attn_decode_multi": (ctypes.c_int, [
        _p, _p, _p, _p, _i32, _p, _p,               # q k v page_table stride seq_lens rel
        _i32, _i32, _i32, _i32, _i32, _i32, _i32,   # B q_len H_q H_kv D page_size num_pages
        _i32, _i32, _f32, _i32,                     # R window scale max_seq_len
        _p, _p, _p, _sz, _i32, _p, _p]),            # out lse ws ws_bytes splits err stream
    "inkling_rel_attn_decode_multi_workspace_size": (_sz, [_i32] * 9),
    "inkling_rel_attn_prefill": (ctypes.c_int, [
        _p, _p, _p, _p, _p, _i32, _p, _p,           # q cu k v page_table stride seq_lens rel
        _i32, _i32, _i32, _i32, _i32, _i32, _i32,   # B T max_q_len H_q H_kv D page_size
        _i32, _i32, _i32, _f32, _i32,               # num_pages R window scale max_seq_len
        _p, _p, _p, _sz, _p, _p]),                  # out lse ws ws_bytes err stream
    "inkling_rel_attn_kv_append": (ctypes.c_int, [
        _p, _p, _p, _p, _p, _i32,                   # k_new v_new cu seq_lens page_table stride
        _i32, _i32, _i32, _i32, _i32, _i32,         # B T H_kv D page_size num_pages
        _p, _p, _p, _p]),                           # k_cache v_cache err stream
    "inkling_rel_attn_kv_conv_append": (ctypes.c_int, [
        _p, _p, _p, _p, _p, _i32,                   # k_new v_new cu seq_lens page_table stride
        _p, _p, _i32, _p, _p, _p, _i32,             # w_k w_v width state_k state_v slots num_slots
        _i32, _i32, _i32, _i32, _i32, _i32, _i32,   # B T max_q_len H_kv D page_size num_pages
        _p, _p, _p, _p]),                           # k_cache v_cache err stream
    "inkling_rel_attn_choose_splits": (_i32, [_i32, _i32, _i32, _i32, _i32]),
    "inkling_rel_attn_decode_workspace_size": (_sz, [_i32] * 8),
    "inkling_rel_attn_prefill_workspace_size": (_sz, [_i32] * 3),
    "inkling_rel_attn_selftest_timeout": (ctypes.c_int, [_p, _i32, _p]),
    "inkling_rel_attn_error_string": (ctypes.c_char_p, [_i32]),
    "inkling_rel_attn_version": (_i32, []),
}


def load():
    """Load the shared library (once) and declare the C signatures."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing; build it first with "
                "paged_attention_relative_attn_gb300.build.build() (needs nvcc)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _v(x):
    return None if x in (None, 0) else int(x)


def inkling_rel_attn_decode(q, k_cache, v_cache, page_table, page_table_stride, seq_lens,
                            rel_logits, B, H_q, H_kv, D, page_size, num_pages, R, window,
                            scale, max_seq_len, out, lse_out, workspace, workspace_bytes,
                            num_splits, device_error, stream):
    return load().inkling_rel_attn_decode(
        _v(q), _v(k_cache), _v(v_cache), _v(page_table), page_table_stride, _v(seq_lens),
        _v(rel_logits), B, H_q, H_kv, D, page_size, num_pages, R, window, scale, max_seq_len,
        _v(out), _v(lse_out), _v(workspace), workspace_bytes, num_splits, _v(device_error),
        _v(stream))


def inkling_rel_attn_decode_noalloc(q, k_cache, v_cache, page_table, page_table_stride, seq_lens,
                                    rel_logits, B, H_q, H_kv, D, page_size, num_pages, R, window,
                                    scale, max_seq_len, out, lse_out, num_splits, device_error,
                                    stream):
    """inkling_rel_attn_decode with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    return load().inkling_rel_attn_decode_noalloc(
        _v(q), _v(k_cache), _v(v_cache), _v(page_table), page_table_stride, _v(seq_lens),
        _v(rel_logits), B, H_q, H_kv, D, page_size, num_pages, R, window, scale, max_seq_len,
        _v(out), _v(lse_out), num_splits, _v(device_error), _v(stream))


def inkling_rel_attn_decode_multi(q, k_cache, v_cache, page_table, page_table_stride, seq_lens,
                                  rel_logits, B, q_len, H_q, H_kv, D, page_size, num_pages, R,
                                  window, scale, max_seq_len, out, lse_out, workspace,
                                  workspace_bytes, num_splits, device_error, stream):
    return load().inkling_rel_attn_decode_multi(
        _v(q), _v(k_cache), _v(v_cache), _v(page_table), page_table_stride, _v(seq_lens),
        _v(rel_logits), B, q_len, H_q, H_kv, D, page_size, num_pages, R, window, scale,
        max_seq_len, _v(out), _v(lse_out), _v(workspace), workspace_bytes, num_splits,
        _v(device_error), _v(stream))


def inkling_rel_attn_decode_multi_workspace_size(B, q_len, H_q, H_kv, D, window, max_seq_len,
                                                 num_splits, num_sms):
    return load().inkling_rel_attn_decode_multi_workspace_size(B, q_len, H_q, H_kv, D, window,
                                                               max_seq_len, num_splits, num_sms)


def inkling_rel_attn_prefill(q, cu_seqlens_q, k_cache, v_cache, page_table, page_table_stride,
                             seq_lens, rel_logits, B, T, max_q_len, H_q, H_kv, D, page_size,
                             num_pages, R, window, scale, max_seq_len, out, lse_out, workspace,
                             workspace_bytes, device_error, stream):
    return load().inkling_rel_attn_prefill(
        _v(q), _v(cu_seqlens_q), _v(k_cache), _v(v_cache), _v(page_table), page_table_stride,
        _v(seq_lens), _v(rel_logits), B, T, max_q_len, H_q, H_kv, D, page_size, num_pages, R,
        window, scale, max_seq_len, _v(out), _v(lse_out), _v(workspace), workspace_bytes,
        _v(device_error), _v(stream))


def inkling_rel_attn_kv_append(k_new, v_new, cu_seqlens_q, seq_lens, page_table,
                               page_table_stride, B, T, H_kv, D, page_size, num_pages, k_cache,
                               v_cache, device_error, stream):
    return load().inkling_rel_attn_kv_append(
        _v(k_new), _v(v_new), _v(cu_seqlens_q), _v(seq_lens), _v(page_table), page_table_stride,
        B, T, H_kv, D, page_size, num_pages, _v(k_cache), _v(v_cache), _v(device_error),
        _v(stream))


def inkling_rel_attn_kv_conv_append(k_new, v_new, cu_seqlens_q, seq_lens, page_table,
                                    page_table_stride, conv_w_k, conv_w_v, width, conv_state_k,
                                    conv_state_v, state_slots, num_slots, B, T, max_q_len, H_kv,
                                    D, page_size, num_pages, k_cache, v_cache, device_error,
                                    stream):
    return load().inkling_rel_attn_kv_conv_append(
        _v(k_new), _v(v_new), _v(cu_seqlens_q), _v(seq_lens), _v(page_table), page_table_stride,
        _v(conv_w_k), _v(conv_w_v), width, _v(conv_state_k), _v(conv_state_v), _v(state_slots),
        num_slots, B, T, max_q_len, H_kv, D, page_size, num_pages, _v(k_cache), _v(v_cache),
        _v(device_error), _v(stream))


def inkling_rel_attn_choose_splits(B, H_kv, window, max_seq_len, num_sms):
    return load().inkling_rel_attn_choose_splits(B, H_kv, window, max_seq_len, num_sms)


def inkling_rel_attn_decode_workspace_size(B, H_q, H_kv, D, window, max_seq_len, num_splits,
                                           num_sms):
    return load().inkling_rel_attn_decode_workspace_size(B, H_q, H_kv, D, window, max_seq_len,
                                                         num_splits, num_sms)


def inkling_rel_attn_prefill_workspace_size(T, H_q, D):
    return load().inkling_rel_attn_prefill_workspace_size(T, H_q, D)


def inkling_rel_attn_selftest_timeout(device_error, timeout_ms, stream):
    return load().inkling_rel_attn_selftest_timeout(_v(device_error), timeout_ms, _v(stream))


def inkling_rel_attn_error_string(code):
    return load().inkling_rel_attn_error_string(code).decode()


def inkling_rel_attn_version():
    return load().inkling_rel_attn_version()
