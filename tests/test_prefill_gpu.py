"""GPU parity of inkling_rel_attn_prefill (through the C ABI) against the CPU
fp64 oracle, plus bit-exact probes and NaN poison."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from oracle.ref import ref_decode
from tests.helpers import assert_close, bits, compact_pages, f64, oracle_prefill

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from paged_attention_relative_attn_gb300 import build
    build.build()
    import paged_attention_relative_attn_gb300 as m
    return m


def run(ops, inp, **kw):
    out, lse = ops.prefill_inputs(inp, **kw)
    torch.cuda.synchronize()
    return out, lse


def make(q_lens, kv_lens, H_q, H_kv, D, P, window, R, seed, q_std=1.0, poison=True, extra_pages=2):
    pool = sum((L + P - 1) // P for L in kv_lens) + extra_pages
    cache = W.make_prefill_cache(kv_lens, H_kv, D, P, device=DEV, seed=seed, pool_pages=pool,
                                 poison=poison)
    return W.make_prefill(cache, q_lens, kv_lens, H_q, R, window, device=DEV, seed=seed + 1,
                          q_std=q_std)


CASES = [
    # q_lens, kv_lens, H_q, H_kv, D, P, window, R
    ([5], [5], 4, 2, 128, 64, 0, 16),
    ([1, 3, 200], [1, 70, 300], 4, 2, 128, 64, 32, 32),
    ([128, 129, 130], [128, 500, 130], 6, 2, 128, 64, 64, 64),
    ([300], [1000], 3, 1, 128, 64, 512, 512),
    ([257, 64], [257, 700], 8, 8, 64, 16, 100, 128),
    ([100, 33], [900, 33], 6, 3, 128, 128, 0, 256),
    ([77], [2000], 4, 1, 128, 32, 0, 1024),
    ([0, 40, 0, 9], [10, 40, 5, 100], 4, 2, 128, 64, 16, 16),
    ([190], [190], 2, 2, 64, 64, 1, 4),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("q_std", [1.0, 4.0])
def test_small_cases(ops, case, q_std):
    ql, kl, H_q, H_kv, D, P, win, R = CASES[case]
    inp = make(ql, kl, H_q, H_kv, D, P, win, R, seed=200 + case, q_std=q_std)
    out, lse = run(ops, inp)
    ro, rl, rows = oracle_prefill(inp)
    idx = torch.tensor(rows, dtype=torch.long, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what=f"case {case}")


@pytest.mark.parametrize("slope", [0.05, 0.3])
def test_rising_bias(ops, slope):
    """rel = -slope * distance: every row's max rises along the key walk, by
    about 4.6 or 28 log2 units per 64-key tile, so the lazy O rescale (taken
    when a row's max passes the exponent base by more than 2^8) runs every one
    to two tiles, each time after waiting for the pending PV."""
    import dataclasses
    inp = make([300, 129], [1000, 400], 6, 2, 128, 64, 0, 1024, seed=260)
    d = torch.arange(inp.R, device=DEV, dtype=torch.float32)
    rel = (-slope * d).expand_as(inp.rel_logits).contiguous()
    inp2 = dataclasses.replace(inp, rel_logits=rel)
    out, lse = run(ops, inp2)
    ro, rl, rows = oracle_prefill(inp2)
    idx = torch.tensor(rows, dtype=torch.long, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what=f"slope {slope}")


def oracle_rows(inp, rows_by_seq):
    """Oracle for selected query rows: row i of sequence b (q_len Q, L keys) is
    the decode query at position L - Q + i over the sequence cut there."""
    cu = inp.cu_seqlens_q.cpu().numpy()
    sl = inp.seq_lens.cpu().numpy()
    outs, lses, toks = [], [], []
    for b, rows in rows_by_seq.items():
        Q = int(cu[b + 1] - cu[b])
        L = int(sl[b])
        for i in rows:
            t = int(cu[b] + i)
            p = L - Q + i
            sel = torch.tensor([b], device=DEV)
            kc, vc, pt, _ = compact_pages(inp.page_table.index_select(0, sel),
                                          torch.tensor([p + 1], device=DEV), inp.page_size,
                                          inp.k_cache, inp.v_cache)
            o, l = ref_decode(f64(inp.q[t:t + 1]), kc, vc, pt, np.array([p + 1]),
                              f64(inp.rel_logits[t:t + 1]), inp.window, inp.scale)
            outs.append(o[0])
            lses.append(l[0])
            toks.append(t)
    return np.stack(outs), np.stack(lses), toks


@pytest.mark.parametrize("chunk", [0, 3])
def test_chunked_prefill_full_size_sampled(ops, chunk):
    """The chunked-prefill workload (4 x 2048 query tokens against the cached
    prefix, window 512, R=512) at full size, checked on sampled rows of every
    128-row tile edge and a few interior rows."""
    inp, _ = W.make_chunked_prefill(chunk, device=DEV, seed=0)
    out, lse = run(ops, inp)
    assert torch.isfinite(out.float()).all()
    rows = {0: [0, 1, 127, 128, 129, 1000, 2047], 1: [5, 511, 512], 2: [255, 256],
            3: [2046, 2047]}
    ro, rl, toks = oracle_rows(inp, rows)
    idx = torch.tensor(toks, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what="chunked")


@pytest.mark.parametrize("chunk", [1, 3])
def test_global_prefill_full_size_sampled(ops, chunk):
    """The global-layer chunked prefill (4 x 2048 query tokens against the
    cached prefix, 8 KV heads, full causal, R = 1024: most distances are past
    the table) at full size, on sampled rows: tile edges, rows whose nearest
    keys cross distance R - 1, and the last row."""
    inp, _ = W.make_chunked_prefill(chunk, device=DEV, seed=0, cfg=W.GLOBAL_PREFILL)
    out, lse = run(ops, inp)
    assert torch.isfinite(out.float()).all()
    rows = {0: [0, 127, 128, 1023, 1024, 2047], 2: [1, 1000], 3: [2046, 2047]}
    ro, rl, toks = oracle_rows(inp, rows)
    idx = torch.tensor(toks, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl,
                 what=f"global prefill call {chunk}")


def test_global_layer_prefill_sampled(ops):
    """A global-layer prefill (full causal, R=1024, distances clamped)."""
    kv = [3000, 1500]
    ql = [700, 1500]
    inp = make(ql, kv, 48, 8, 128, 64, 0, 1024, seed=5, poison=False)
    out, lse = run(ops, inp)
    rows = {0: [0, 1, 128, 350, 699], 1: [0, 1, 127, 1023, 1024, 1499]}
    ro, rl, toks = oracle_rows(inp, rows)
    idx = torch.tensor(toks, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what="global")


def permuted(inp, seed):
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(inp.num_pages, generator=g).to(DEV)
    kc = torch.empty_like(inp.k_cache)
    vc = torch.empty_like(inp.v_cache)
    kc[perm] = inp.k_cache
    vc[perm] = inp.v_cache
    return W.PrefillInputs(q=inp.q, cu_seqlens_q=inp.cu_seqlens_q, k_cache=kc, v_cache=vc,
                           page_table=perm[inp.page_table.long()].to(torch.int32),
                           seq_lens=inp.seq_lens, rel_logits=inp.rel_logits, window=inp.window,
                           scale=inp.scale, max_seq_len=inp.max_seq_len, max_q_len=inp.max_q_len)


def test_page_permutation_bit_exact(ops):
    inp = make([300, 129], [1000, 129], 6, 2, 128, 64, 512, 512, seed=9)
    out0, lse0 = run(ops, inp)
    for s in range(3):
        out1, lse1 = run(ops, permuted(inp, 70 + s))
        assert np.array_equal(bits(out0), bits(out1))
        assert torch.equal(lse0, lse1)


@pytest.mark.parametrize("P", [64, 16])
def test_one_hot_bias_bit_exact(ops, P):
    """rel = -1e4 except at distance d*: every query row must output the bf16
    V row of key p - d* exactly (or 0-weight rows for p < d*)."""
    ql, kl = [200, 70], [600, 70]
    inp = make(ql, kl, 4, 2, 128, P, 128, 128, seed=11, poison=False)
    cu = inp.cu_seqlens_q.cpu().tolist()
    pt = inp.page_table.cpu()
    for d in [0, 1, 3, 63, 64, 65, 127]:
        rel = torch.full_like(inp.rel_logits, -1e4)
        rel[:, :, d] = 0.0
        inp2 = W.PrefillInputs(q=inp.q, cu_seqlens_q=inp.cu_seqlens_q, k_cache=inp.k_cache,
                               v_cache=inp.v_cache, page_table=inp.page_table,
                               seq_lens=inp.seq_lens, rel_logits=rel, window=inp.window,
                               scale=inp.scale, max_seq_len=inp.max_seq_len,
                               max_q_len=inp.max_q_len)
        out, _ = run(ops, inp2)
        for b, (Q, L) in enumerate(zip(ql, kl)):
            for i in range(0, Q, 7):
                p = L - Q + i
                if p - d < 0:
                    continue
                j = p - d
                page, slot = int(pt[b, j // P]), j % P
                t = cu[b] + i
                want = inp.v_cache[page, slot]  # [H_kv, D]
                got = out[t]
                for h in range(4):
                    assert torch.equal(got[h], want[h // 2]), (d, b, i, h)


def test_nan_poison_and_output_reuse(ops):
    inp = make([150, 60], [800, 60], 6, 2, 128, 64, 512, 512, seed=12, poison=True)
    out = torch.full_like(inp.q, float("nan"))
    run(ops, inp, out=out)
    ro, rl, rows = oracle_prefill(inp)
    idx = torch.tensor(rows, dtype=torch.long, device=DEV)
    assert_close(out.index_select(0, idx), ro, what="poison")


def test_bad_chunk_reported(ops):
    inp = make([10], [20], 4, 2, 128, 64, 0, 16, seed=13)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bad = W.PrefillInputs(q=inp.q, cu_seqlens_q=inp.cu_seqlens_q, k_cache=inp.k_cache,
                          v_cache=inp.v_cache, page_table=inp.page_table,
                          seq_lens=torch.tensor([5], dtype=torch.int32, device=DEV),
                          rel_logits=inp.rel_logits, window=0, scale=inp.scale,
                          max_seq_len=20, max_q_len=10)
    run(ops, bad, device_error=err)
    assert int(err.item()) & 8
