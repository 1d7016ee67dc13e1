"""PyTorch-facing wrappers: shape/dtype checks, default output buffers, the
current stream, then one call into the C ABI.  All arithmetic happens in the
CUDA kernels of libinkling_rel_attn.so; there is no CPU or PyTorch fallback.
"""

from __future__ import annotations

import torch

from . import _lib


class InklingError(RuntimeError):
    """A non-zero INKLING_* status from the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_lib.inkling_rel_attn_error_string(code)} (code {code})")


def _check(rc: int, where: str):
    if rc != 0:
        raise InklingError(rc, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _need(t, name, dtype, dims):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.dim() != dims:
        raise ValueError(f"{name}: expected {dims} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def choose_splits(B, H_kv, window, max_seq_len, num_sms=0):
    return _lib.inkling_rel_attn_choose_splits(B, H_kv, window, max_seq_len, num_sms)


def decode_workspace_bytes(B, H_q, H_kv, D, window, max_seq_len, num_splits=0, num_sms=0):
    return _lib.inkling_rel_attn_decode_workspace_size(B, H_q, H_kv, D, window, max_seq_len,
                                                       num_splits, num_sms)


def decode(q, k_cache, v_cache, page_table, seq_lens, rel_logits, *, window, scale,
           max_seq_len, out=None, lse=None, workspace=None, num_splits=0,
           device_error=None, stream=None):
    """Decode attention (one query per sequence).  See inkling_rel_attn_decode.

    q [B, H_q, D] bf16; k_cache, v_cache [num_pages, page_size, H_kv, D] bf16;
    page_table [B, stride] int32; seq_lens [B] int32; rel_logits [B, H_q, R] fp32.
    Returns (out bf16 [B, H_q, D], lse fp32 [B, H_q]).  Pass ``out``, ``lse`` and
    ``workspace`` to avoid allocations (required under CUDA-graph capture).
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(rel_logits, "rel_logits", torch.float32, 3)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    B, H_q, D = q.shape
    num_pages, P, H_kv, Dk = k_cache.shape
    R = rel_logits.shape[2]
    if Dk != D or rel_logits.shape[:2] != (B, H_q) or seq_lens.shape[0] != B or page_table.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=q.device)
    ws_need = decode_workspace_bytes(B, H_q, H_kv, D, window, max_seq_len, num_splits)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.inkling_rel_attn_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.shape[1],
        _ptr(seq_lens), _ptr(rel_logits), B, H_q, H_kv, D, P, num_pages, R, window,
        float(scale), max_seq_len, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        num_splits, _ptr(device_error), _stream(q.device, stream))
    _check(rc, "inkling_rel_attn_decode")
    return out, lse


def decode_multi_workspace_bytes(B, q_len, H_q, H_kv, D, window, max_seq_len, num_splits=0,
                                 num_sms=0):
    return _lib.inkling_rel_attn_decode_multi_workspace_size(B, q_len, H_q, H_kv, D, window,
                                                             max_seq_len, num_splits, num_sms)


def decode_multi(q, k_cache, v_cache, page_table, seq_lens, rel_logits, *, q_len, window, scale,
                 max_seq_len, out=None, lse=None, workspace=None, num_splits=0,
                 device_error=None, stream=None):
    """Decode of ``q_len`` new tokens per sequence (the last q_len of each).
    See inkling_rel_attn_decode_multi.

    q [B * q_len, H_q, D] bf16 (row b * q_len + i); rel_logits [B * q_len, H_q, R]
    fp32; other tensors as ``decode``.  Returns (out [B * q_len, H_q, D] bf16,
    lse [B * q_len, H_q] fp32).
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(rel_logits, "rel_logits", torch.float32, 3)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    T, H_q, D = q.shape
    B = seq_lens.shape[0]
    num_pages, P, H_kv, Dk = k_cache.shape
    R = rel_logits.shape[2]
    if (Dk != D or T != B * q_len or rel_logits.shape[:2] != (T, H_q)
            or page_table.shape[0] != B):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, H_q), dtype=torch.float32, device=q.device)
    ws_need = decode_multi_workspace_bytes(B, q_len, H_q, H_kv, D, window, max_seq_len, num_splits)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.inkling_rel_attn_decode_multi(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.shape[1],
        _ptr(seq_lens), _ptr(rel_logits), B, q_len, H_q, H_kv, D, P, num_pages, R, window,
        float(scale), max_seq_len, _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
        num_splits, _ptr(device_error), _stream(q.device, stream))
    _check(rc, "inkling_rel_attn_decode_multi")
    return out, lse


def prefill(q, cu_seqlens_q, k_cache, v_cache, page_table, seq_lens, rel_logits, *, window,
            scale, max_seq_len, max_q_len, out=None, lse=None, device_error=None, stream=None):
    """Chunked / paged prefill.  See inkling_rel_attn_prefill.

    q [T, H_q, D] bf16; cu_seqlens_q [B+1] int32; rel_logits [T, H_q, R] fp32.
    Returns (out bf16 [T, H_q, D], lse fp32 [T, H_q]).
    """
    _need(q, "q", torch.bfloat16, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(rel_logits, "rel_logits", torch.float32, 3)
    T, H_q, D = q.shape
    num_pages, P, H_kv, _ = k_cache.shape
    B = seq_lens.shape[0]
    R = rel_logits.shape[2]
    if cu_seqlens_q.shape[0] != B + 1 or rel_logits.shape[:2] != (T, H_q):
        raise ValueError("inconsistent shapes")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, H_q), dtype=torch.float32, device=q.device)
    rc = _lib.inkling_rel_attn_prefill(
        _ptr(q), _ptr(cu_seqlens_q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
        page_table.shape[1], _ptr(seq_lens), _ptr(rel_logits), B, T, max_q_len, H_q, H_kv, D, P,
        num_pages, R, window, float(scale), max_seq_len, _ptr(out), _ptr(lse), None, 0,
        _ptr(device_error), _stream(q.device, stream))
    _check(rc, "inkling_rel_attn_prefill")
    return out, lse


def kv_append(k_new, v_new, cu_seqlens_q, seq_lens, page_table, k_cache, v_cache, *,
              device_error=None, stream=None):
    """Write the new tokens' K/V into the paged cache (in place).  See
    inkling_rel_attn_kv_append.

    k_new, v_new [T, H_kv, D] bf16; cu_seqlens_q [B+1] int32; seq_lens [B]
    int32 (totals including the new tokens); page_table [B, stride] int32;
    k_cache, v_cache [num_pages, page_size, H_kv, D] bf16, updated in place.
    """
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(page_table, "page_table", torch.int32, 2)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    T, H_kv, D = k_new.shape
    num_pages, P, H_kv_c, D_c = k_cache.shape
    B = seq_lens.shape[0]
    if (v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or (H_kv_c, D_c) != (H_kv, D)
            or cu_seqlens_q.shape[0] != B + 1 or page_table.shape[0] != B):
        raise ValueError("inconsistent shapes")
    rc = _lib.inkling_rel_attn_kv_append(
        _ptr(k_new), _ptr(v_new), _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(page_table),
        page_table.shape[1], B, T, H_kv, D, P, num_pages, _ptr(k_cache), _ptr(v_cache),
        _ptr(device_error), _stream(k_new.device, stream))
    _check(rc, "inkling_rel_attn_kv_append")


def kv_conv_append(k_new, v_new, cu_seqlens_q, seq_lens, page_table, k_cache, v_cache,
                   conv_w_k, conv_w_v, conv_state_k, conv_state_v, state_slots, *,
                   max_q_len, device_error=None, stream=None):
    """The causal short convolutions on K and V of the new tokens, then the
    append of the convolved rows into the paged cache; the state pool rows of
    the sequences are rewritten in place.  See inkling_rel_attn_kv_conv_append.

    k_new, v_new [T, H_kv, D] bf16; conv_w_k, conv_w_v [H_kv, D, width] fp32;
    conv_state_k, conv_state_v [num_slots, width - 1, H_kv, D] bf16 (width 1:
    None); state_slots [B] int32; the rest as for ``kv_append``.  max_q_len is
    a host bound on any sequence's new tokens.
    """
    _need(k_new, "k_new", torch.bfloat16, 3)
    _need(v_new, "v_new", torch.bfloat16, 3)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(page_table, "page_table", torch.int32, 2)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(conv_w_k, "conv_w_k", torch.float32, 3)
    _need(conv_w_v, "conv_w_v", torch.float32, 3)
    T, H_kv, D = k_new.shape
    num_pages, P, H_kv_c, D_c = k_cache.shape
    B = seq_lens.shape[0]
    width = conv_w_k.shape[2]
    if (v_new.shape != k_new.shape or v_cache.shape != k_cache.shape or (H_kv_c, D_c) != (H_kv, D)
            or cu_seqlens_q.shape[0] != B + 1 or page_table.shape[0] != B
            or tuple(conv_w_k.shape) != (H_kv, D, width) or conv_w_v.shape != conv_w_k.shape):
        raise ValueError("inconsistent shapes")
    num_slots = 0
    if width > 1:
        _need(conv_state_k, "conv_state_k", torch.bfloat16, 4)
        _need(conv_state_v, "conv_state_v", torch.bfloat16, 4)
        _need(state_slots, "state_slots", torch.int32, 1)
        num_slots = conv_state_k.shape[0]
        if (tuple(conv_state_k.shape) != (num_slots, width - 1, H_kv, D)
                or conv_state_v.shape != conv_state_k.shape or state_slots.shape[0] != B):
            raise ValueError("inconsistent state shapes")
    rc = _lib.inkling_rel_attn_kv_conv_append(
        _ptr(k_new), _ptr(v_new), _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(page_table),
        page_table.shape[1], _ptr(conv_w_k), _ptr(conv_w_v), width, _ptr(conv_state_k),
        _ptr(conv_state_v), _ptr(state_slots), num_slots, B, T, int(max_q_len), H_kv, D, P,
        num_pages, _ptr(k_cache), _ptr(v_cache), _ptr(device_error), _stream(k_new.device, stream))
    _check(rc, "inkling_rel_attn_kv_conv_append")


def decode_inputs(inp, **kw):
    """``decode`` on a workloads.DecodeInputs-like object."""
    return decode(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_lens, inp.rel_logits,
                  window=inp.window, scale=inp.scale, max_seq_len=inp.max_seq_len, **kw)


def prefill_inputs(inp, **kw):
    """``prefill`` on a workloads.PrefillInputs-like object."""
    return prefill(inp.q, inp.cu_seqlens_q, inp.k_cache, inp.v_cache, inp.page_table,
                   inp.seq_lens, inp.rel_logits, window=inp.window, scale=inp.scale,
                   max_seq_len=inp.max_seq_len, max_q_len=inp.max_q_len, **kw)
