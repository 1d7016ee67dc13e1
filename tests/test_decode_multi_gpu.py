"""Multi-token decode (q_len new tokens per sequence) through the C ABI
against the oracle.  The oracle is the prefill definition with q_len query
tokens per sequence (the last q_len tokens, packed row b * q_len + i)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_close, bits, oracle_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    import paged_attention_relative_attn_gb300 as ira
    from paged_attention_relative_attn_gb300 import build
    build.build()
    return ira


def make(B_lens, q_len, H_q, H_kv, D, P, window, R, seed, poison=True):
    cache = W.make_prefill_cache(B_lens, H_kv, D, P, device=DEV, seed=seed,
                                 pool_pages=sum(W.pages_for(L, P) for L in B_lens) + 2,
                                 poison=poison)
    return W.make_prefill(cache, [q_len] * len(B_lens), B_lens, H_q, R, window, device=DEV,
                          seed=seed + 1)


def run(ops, inp, q_len, **kw):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = ops.decode_multi(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_lens,
                                inp.rel_logits, q_len=q_len, window=inp.window, scale=inp.scale,
                                max_seq_len=inp.max_seq_len, device_error=err, **kw)
    torch.cuda.synchronize()
    return out, lse, int(err.item())


CASES = [
    # lens, q_len, H_q, H_kv, D, P, window, R
    ([9, 64, 200, 1000], 2, 12, 4, 128, 64, 32, 32),     # G=3, one group of 2
    ([5, 70, 513, 2000], 4, 12, 4, 128, 16, 0, 256),      # G=3, full causal, clamp
    ([8, 100, 700], 8, 12, 4, 128, 64, 64, 64),           # G=3: groups of 5 + 3
    ([3, 40, 300], 3, 12, 2, 64, 16, 16, 16),             # G=6: groups of 2 + 1, D=64
    ([8, 9, 129, 4000], 8, 12, 2, 128, 64, 0, 1024),      # G=6: four groups, long causal
    ([6, 50], 6, 4, 4, 128, 64, 5, 8),                    # G=1: groups of 6, tiny window
    ([16, 33], 5, 16, 1, 64, 16, 0, 64),                  # G=16: groups of 1
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_small_cases(ops, case):
    lens, ql, H_q, H_kv, D, P, win, R = CASES[case]
    inp = make(lens, ql, H_q, H_kv, D, P, win, R, seed=300 + case)
    out, lse, err = run(ops, inp, ql)
    assert err == 0
    ro, rl, _ = oracle_prefill(inp)
    assert_close(out, ro, lse, rl, what=f"case {case}")


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_forced_splits(ops, splits):
    """Splits of a sequence's keys, merged by log-sum-exp; an early token
    group has fewer keys than the last, so some of its splits are empty."""
    lens, ql, H_q, H_kv, D, P, win, R = CASES[4]
    inp = make(lens, ql, H_q, H_kv, D, P, win, R, seed=350 + splits)
    out, lse, err = run(ops, inp, ql, num_splits=splits)
    assert err == 0
    ro, rl, _ = oracle_prefill(inp)
    assert_close(out, ro, lse, rl, what=f"{splits} splits")


@pytest.mark.parametrize("case,splits", [(1, 3), (1, 7), (2, 2)])
def test_forced_splits_six_rows(ops, case, splits):
    """Token groups of 2 tokens x 3 heads (six rows, D = 128: the two-round
    item combine) over splits of long causal ranges; an early group sees
    fewer keys than the last, so a split can be empty for it."""
    lens, ql, H_q, H_kv, D, P, win, R = CASES[case]
    inp = make(lens, ql, H_q, H_kv, D, P, win, R, seed=370 + 10 * case + splits)
    out, lse, err = run(ops, inp, ql, num_splits=splits)
    assert err == 0
    ro, rl, _ = oracle_prefill(inp)
    assert_close(out, ro, lse, rl, what=f"case {case}, {splits} splits")


@pytest.mark.parametrize("slope", [0.05, 0.3])
def test_rising_bias(ops, slope):
    """rel = -slope * distance: every row's max rises along the key walk, so
    the lazily re-reduced exponent base and the O rescale are taken every one
    to two tiles (two n-tiles: 4 tokens x 3 heads per item)."""
    import dataclasses
    lens, ql = [700, 1000, 129, 64], 4
    inp = make(lens, ql, 12, 4, 128, 64, 512, 512, seed=390)
    d = torch.arange(inp.R, device=DEV, dtype=torch.float32)
    rel = (-slope * d).expand_as(inp.rel_logits).contiguous()
    inp2 = dataclasses.replace(inp, rel_logits=rel)
    out, lse, err = run(ops, inp2, ql)
    assert err == 0
    ro, rl, tok = oracle_prefill(inp2)
    assert_close(out, ro, lse, rl, what=f"slope {slope}")


def test_one_token_is_decode_bit_exact(ops):
    inp = W.make_decode(6, 48, 16, 128, 64, [1, 63, 64, 65, 700, 3000], 512, 512, device=DEV,
                        seed=21)
    ref_out, ref_lse = ops.decode_inputs(inp)
    out, lse = ops.decode_multi(inp.q, inp.k_cache, inp.v_cache, inp.page_table, inp.seq_lens,
                                inp.rel_logits, q_len=1, window=inp.window, scale=inp.scale,
                                max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(ref_out))
    assert torch.equal(lse, ref_lse)


def test_sequence_shorter_than_q_len(ops):
    """seq_lens[b] < q_len cannot hold the q_len new tokens: reported, and
    those tokens get out = 0, lse = -inf; the other sequences are exact."""
    inp = make([30, 40], 4, 12, 4, 128, 64, 0, 64, seed=7, poison=False)
    inp.seq_lens[0] = 2
    out, lse, err = run(ops, inp, 4)
    assert err & 8  # INKLING_DEVERR_BAD_CHUNK
    assert torch.all(out[:4] == 0) and torch.all(torch.isneginf(lse[:4]))
    ro, rl, rows = oracle_prefill(inp, [1])
    idx = torch.tensor(rows, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what="second")


def test_full_size_sampled(ops):
    """The multi-token local decode workload (64 sequences x 4 new tokens,
    48/16 heads, window 512, R = 512), oracle on sampled sequences."""
    lens = W.draw_uniform_lengths(64, 1024, 8192, 0)
    inp = make(lens, 4, 48, 16, 128, 64, 512, 512, seed=0, poison=False)
    out, lse, err = run(ops, inp, 4)
    assert err == 0
    seqs = [0, 17, 63]
    ro, rl, rows = oracle_prefill(inp, seqs)
    idx = torch.tensor(rows, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what="full size")
