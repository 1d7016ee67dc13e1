"""inkling_rel_attn_decode_noalloc: decode for callers that cannot allocate
device memory (a plugin inside a framework that owns all device memory, a
binding without access to the CUDA allocator).  Its split partials live in a
fixed scratch array inside the library; this checks, through the C ABI, that
two consecutive calls give bit for bit the result of the regular entry point
with a caller workspace (same kernels, same split plan), and the oracle's on
sampled sequences.  Collected last (file name) so that a run stopping at the
first failure has already run every other test."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_close, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_attention_relative_attn_gb300 import build, _lib
    build.build()
    return _lib


def _args(inp):
    return dict(q=inp.q.data_ptr(), k_cache=inp.k_cache.data_ptr(), v_cache=inp.v_cache.data_ptr(),
                page_table=inp.page_table.data_ptr(), page_table_stride=inp.page_table.shape[1],
                seq_lens=inp.seq_lens.data_ptr(), rel_logits=inp.rel_logits.data_ptr(), B=inp.B,
                H_q=inp.H_q, H_kv=inp.H_kv, D=inp.D, page_size=inp.page_size,
                num_pages=inp.num_pages, R=inp.R, window=inp.window, scale=inp.scale,
                max_seq_len=inp.max_seq_len)


def _regular(lib, inp, splits):
    out = torch.empty_like(inp.q)
    lse = torch.empty(inp.q.shape[:2], device="cuda")
    need = lib.inkling_rel_attn_decode_workspace_size(inp.B, inp.H_q, inp.H_kv, inp.D, inp.window,
                                                      inp.max_seq_len, splits, 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    rc = lib.inkling_rel_attn_decode(**_args(inp), out=out.data_ptr(), lse_out=lse.data_ptr(),
                                     workspace=ws.data_ptr(), workspace_bytes=ws.numel(),
                                     num_splits=splits, device_error=None,
                                     stream=torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    return out, lse


def _noalloc(lib, inp, splits):
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full(inp.q.shape[:2], float("nan"), device="cuda")
    rc = lib.inkling_rel_attn_decode_noalloc(**_args(inp), out=out.data_ptr(),
                                             lse_out=lse.data_ptr(), num_splits=splits,
                                             device_error=None,
                                             stream=torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    return out, lse


def test_noalloc_matches_regular_on_two_calls(lib):
    # two different global-layer batches (full causal, R = 1024, split-KV), so
    # the second call reuses scratch the first one filled
    cases = [W.make_decode(8, 48, 8, 128, 64, [20000, 1, 4096, 777, 12000, 65, 3000, 9999], 0,
                           1024, device="cuda", seed=41, max_seq_len=20000),
             W.make_decode(6, 48, 8, 128, 64, [5000, 30000, 2, 640, 17000, 8191], 0, 1024,
                           device="cuda", seed=42, max_seq_len=30000)]
    for inp in cases:
        # the call splits its keys, so its partials go through the shared array
        need = lib.inkling_rel_attn_decode_workspace_size(inp.B, inp.H_q, inp.H_kv, inp.D,
                                                          inp.window, inp.max_seq_len, 0, 0)
        assert need > 0
        ref_out, ref_lse = _regular(lib, inp, 0)
        out, lse = _noalloc(lib, inp, 0)
        torch.cuda.synchronize()
        # same kernels and the same split plan: identical bits, whatever the
        # array held before
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        # and the oracle agrees on sampled sequences
        sample = [0, 1, inp.B - 1]
        ro, rl = oracle_decode(inp, sample)
        idx = torch.tensor(sample, device="cuda")
        assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what="noalloc")


def test_noalloc_rejects_calls_beyond_its_scratch(lib):
    inp = W.make_decode(2, 48, 8, 128, 64, [100, 200], 0, 64, device="cuda", seed=43,
                        max_seq_len=200)
    big = dict(_args(inp), B=4096, max_seq_len=1 << 20)  # needs far more than 32 MiB
    out = torch.empty_like(inp.q)
    rc = lib.inkling_rel_attn_decode_noalloc(**big, out=out.data_ptr(), lse_out=None,
                                             num_splits=128, device_error=None,
                                             stream=torch.cuda.current_stream().cuda_stream)
    assert rc == -3
