"""Guard regions around every attention output and the decode workspace.

Each buffer the library writes (out, lse, the split workspace) sits inside
one larger allocation with guard bytes of a fixed pattern before and after
it; the call must leave every guard byte as it was and overwrite every
element it owns.  Prefill calls also leave rows of `out` / `lse` that belong
to no sequence (past cu_seqlens_q[B]) untouched, with query tiles that end
mid-tile (the partial-tile epilogue) and full tiles (the TMA-store
epilogue).  Decode output reuse across calls is the other half of this
(test_decode_gpu.test_output_reuse_and_empty_sequences)."""

from __future__ import annotations

import math

import pytest
import torch

import workloads as W
from tests.helpers import assert_close, oracle_decode, oracle_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096       # bytes of guard before and after each buffer
PATTERN = 0xA5     # guard byte (bf16 0xA5A5 and fp32 0xA5A5A5A5 are finite, distinctive)


@pytest.fixture(scope="module")
def ops():
    import paged_attention_relative_attn_gb300 as ira
    from paged_attention_relative_attn_gb300 import build
    build.build()
    return ira


class Guarded:
    """A `shape` tensor of `dtype` at byte offset GUARD of one allocation with
    GUARD bytes of PATTERN on both sides; the tensor itself is filled with
    `fill` (NaN by default) so that an element the call fails to write shows."""

    def __init__(self, shape, dtype, fill=float("nan")):
        esize = torch.empty((), dtype=dtype).element_size()
        self.n = math.prod(shape) * esize
        self.buf = torch.full((2 * GUARD + self.n,), PATTERN, dtype=torch.uint8, device=DEV)
        self.t = self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def intact(self):
        return bool((self.buf[:GUARD] == PATTERN).all()) and \
            bool((self.buf[GUARD + self.n:] == PATTERN).all())


def _workspace(nbytes):
    """Workspace of exactly `nbytes` inside guards (its contents are the
    library's own scratch: only the guards are checked)."""
    return Guarded((max(nbytes, 16),), torch.uint8, fill=None)


@pytest.mark.parametrize("case", ["local", "global_split", "global_forced", "tiny_d64"])
def test_decode_writes_only_its_buffers(ops, case):
    if case == "local":
        inp = W.make_decode(9, 48, 16, 128, 64, [1, 63, 64, 65, 511, 512, 513, 3000, 8192], 512,
                            512, device=DEV, seed=301)
        splits = 0
    elif case == "global_split":
        inp = W.make_decode(6, 48, 8, 128, 64, [20000, 1, 4097, 64, 9000, 2], 0, 1024,
                            device=DEV, seed=302)
        splits = 0
    elif case == "global_forced":
        inp = W.make_decode(5, 48, 8, 128, 64, [4096, 1, 777, 3000, 2049], 0, 1024, device=DEV,
                            seed=303)
        splits = 7
    else:
        # D = 64, pages of 16, full causal: three splits of the 300 keys
        inp = W.make_decode(3, 4, 2, 64, 16, [37, 100, 300], 0, 32, device=DEV, seed=304,
                            poison=True, pool_pages=40)
        splits = 3
    need = ops.decode_workspace_bytes(inp.B, inp.H_q, inp.H_kv, inp.D, inp.window,
                                      inp.max_seq_len, splits)
    if case != "local":
        assert need > 0  # the call goes through the workspace
    out = Guarded(tuple(inp.q.shape), torch.bfloat16)
    lse = Guarded((inp.B, inp.H_q), torch.float32)
    ws = _workspace(need)
    ops.decode_inputs(inp, out=out.t, lse=lse.t, workspace=ws.t[:need] if need else None,
                      num_splits=splits)
    torch.cuda.synchronize()
    assert out.intact() and lse.intact() and ws.intact(), case
    ro, rl = oracle_decode(inp)
    assert_close(out.t, ro, lse.t, rl, what=case)


def test_decode_multi_writes_only_its_buffers(ops):
    lens = [8, 100, 700, 4000, 5]
    q_len = 4
    cache = W.make_prefill_cache(lens, 8, 128, 64, device=DEV, seed=311)
    inp = W.make_prefill(cache, [q_len] * len(lens), lens, 48, 1024, 0, device=DEV, seed=312)
    for splits in (0, 5):
        need = ops.decode_multi_workspace_bytes(len(lens), q_len, 48, 8, 128, 0, inp.max_seq_len,
                                                splits)
        out = Guarded(tuple(inp.q.shape), torch.bfloat16)
        lse = Guarded(tuple(inp.q.shape[:2]), torch.float32)
        ws = _workspace(need)
        ops.decode_multi(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_lens,
                         inp.rel_logits, q_len=q_len, window=0, scale=inp.scale,
                         max_seq_len=inp.max_seq_len, out=out.t, lse=lse.t,
                         workspace=ws.t[:need] if need else None, num_splits=splits)
        torch.cuda.synchronize()
        assert out.intact() and lse.intact() and ws.intact(), splits
        ro, rl, rows = oracle_prefill(inp)
        idx = torch.tensor(rows, device=DEV)
        assert_close(out.t.index_select(0, idx), ro, lse.t.index_select(0, idx), rl,
                     what=f"multi splits={splits}")


PREFILL = [
    # q_lens, kv_lens, H_q, H_kv, D, P, window, R, spare rows past cu_seqlens_q[B]
    ([128, 256], [128, 900], 6, 2, 128, 64, 0, 256, 40),        # full tiles only
    ([130, 1, 255, 129], [130, 70, 300, 2000], 6, 2, 128, 64, 64, 64, 7),  # partial tiles
    ([77, 300], [1000, 300], 4, 1, 64, 16, 32, 32, 128),        # D = 64, row-by-row stores
    ([2048, 100], [4096, 100], 48, 16, 128, 64, 512, 512, 200),  # many tiles, window
]


@pytest.mark.parametrize("case", range(len(PREFILL)))
def test_prefill_writes_only_its_rows(ops, case):
    ql, kl, H_q, H_kv, D, P, win, R, spare = PREFILL[case]
    cache = W.make_prefill_cache(kl, H_kv, D, P, device=DEV, seed=320 + case,
                                 pool_pages=sum(W.pages_for(L, P) for L in kl) + 2, poison=True)
    inp = W.make_prefill(cache, ql, kl, H_q, R, win, device=DEV, seed=330 + case)
    T = inp.T
    Tx = T + spare  # rows T .. Tx-1 of the buffers belong to no sequence
    q = torch.zeros((Tx, H_q, D), dtype=torch.bfloat16, device=DEV)
    q[:T] = inp.q
    rel = torch.zeros((Tx, H_q, R), dtype=torch.float32, device=DEV)
    rel[:T] = inp.rel_logits
    out = Guarded((Tx, H_q, D), torch.bfloat16)
    lse = Guarded((Tx, H_q), torch.float32)
    ops.prefill(q, inp.cu_seqlens_q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_lens, rel,
                window=win, scale=inp.scale, max_seq_len=inp.max_seq_len,
                max_q_len=inp.max_q_len, out=out.t, lse=lse.t)
    torch.cuda.synchronize()
    assert out.intact() and lse.intact()
    # rows past the last sequence keep their NaN fill, bit for bit
    nan_bf16 = torch.full((1,), float("nan"), dtype=torch.bfloat16, device=DEV).view(torch.int16)
    assert torch.all(out.t[T:].view(torch.int16) == nan_bf16)
    assert torch.all(torch.isnan(lse.t[T:]))
    ro, rl, rows = oracle_prefill(inp)
    idx = torch.tensor(rows, device=DEV)
    assert_close(out.t.index_select(0, idx), ro, lse.t.index_select(0, idx), rl,
                 what=f"prefill case {case}")
