"""GPU parity of inkling_rel_attn_decode (through the C ABI) against the CPU
fp64 oracle, bit-exact probes, split/merge agreement, graph capture, NaN
poison, output reuse and device-side error reporting."""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_close, bits, oracle_decode

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    from paged_attention_relative_attn_gb300 import build
    build.build()
    import paged_attention_relative_attn_gb300 as m
    return m


def run(ops, inp, **kw):
    out, lse = ops.decode_inputs(inp, **kw)
    torch.cuda.synchronize()
    return out, lse


# ------------------------------------------------------------------ parity
def test_tiny_decode(ops):
    inp = W.make_decode_config("tiny_decode", device=DEV)
    out, lse = run(ops, inp)
    ro, rl = oracle_decode(inp)
    assert_close(out, ro, lse, rl, what="tiny_decode")


@pytest.mark.parametrize("name,sample", [("local_decode", [0, 5, 17, 31, 42, 63]),
                                         ("global_decode", [0, 9, 21, 31])])
def test_full_size_sampled(ops, name, sample):
    """The bench's configuration (auto split count), checked on sampled
    sequences by the oracle."""
    inp = W.make_decode_config(name, device=DEV)
    out, lse = run(ops, inp)
    ro, rl = oracle_decode(inp, sample)
    idx = torch.tensor(sample, device=DEV)
    assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl, what=name)
    assert torch.isfinite(out.float()).all()


SMALL = [
    # lens, H_q, H_kv, D, P, window, R
    ([1, 63, 64, 65, 127, 128, 129], 6, 2, 128, 64, 0, 128),
    ([31, 32, 33, 100, 511, 512, 513], 48, 16, 128, 64, 512, 512),
    ([1, 15, 16, 17, 200], 4, 2, 64, 16, 32, 32),
    ([300, 257, 1000], 8, 8, 128, 32, 0, 64),
    ([700, 129, 64, 3], 16, 1, 64, 128, 100, 40),
    ([2000, 1500], 48, 8, 128, 64, 0, 1024),
    ([513, 1025, 2049], 12, 4, 128, 64, 0, 7),
    ([0, 5, 0, 70], 6, 1, 128, 64, 64, 64),
    ([90], 3, 3, 64, 16, 1, 4),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
@pytest.mark.parametrize("q_std", [1.0, 4.0])
def test_small_cases(ops, case, q_std):
    lens, H_q, H_kv, D, P, win, R = SMALL[case]
    pool = sum((L + P - 1) // P for L in lens) + 3
    inp = W.make_decode(len(lens), H_q, H_kv, D, P, lens, win, R, device=DEV, seed=100 + case,
                        pool_pages=pool, poison=True, q_std=q_std)
    out, lse = run(ops, inp)
    ro, rl = oracle_decode(inp)
    assert_close(out, ro, lse, rl, what=f"case {case}")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 16, 128])
def test_forced_splits(ops, splits):
    lens = [4096, 1, 777, 3000, 2049]
    inp = W.make_decode(len(lens), 48, 8, 128, 64, lens, 0, 1024, device=DEV, seed=7,
                        poison=True, q_std=3.0)
    ref_out, ref_lse = run(ops, inp, num_splits=1)
    out, lse = run(ops, inp, num_splits=splits)
    # splits change only the fp32 reduction order
    assert (out.float() - ref_out.float()).abs().max().item() <= 1.6e-2
    assert (lse - ref_lse).abs().max().item() <= 1e-4
    ro, rl = oracle_decode(inp)
    assert_close(out, ro, lse, rl, what=f"splits={splits}")


def test_decode_66_layers_every_layer(ops):
    """The 66-layer decode step exactly as the benchmark draws it (batch 128,
    lognormal lengths, layer l from seed 1000 + l, global iff l % 6 == 5),
    every layer at full size, each checked by the oracle on three sampled
    sequences (one of them the layer's longest)."""
    lens = W.draw_stack_lengths(0)
    s = W.STACK
    longest = int(np.argmax(lens))
    n_global = 0
    for layer in range(s["n_layers"]):
        c = s["glob"] if W.is_global_layer(layer) else s["local"]
        n_global += W.is_global_layer(layer)
        inp = W.make_decode(s["B"], s["H_q"], c["H_kv"], s["D"], s["P"], lens, c["window"],
                            c["R"], device=DEV, seed=1000 + layer, max_seq_len=s["max_len"])
        out, lse = run(ops, inp)
        sample = sorted({layer % s["B"], (37 * layer + 11) % s["B"], longest})
        ro, rl = oracle_decode(inp, sample)
        idx = torch.tensor(sample, device=DEV)
        assert_close(out.index_select(0, idx), ro, lse.index_select(0, idx), rl,
                     what=f"layer {layer}")
        assert torch.isfinite(out.float()).all(), layer
        del inp, out, lse
    assert n_global == 11


# ------------------------------------------------------------------ bit-exact
def permuted_copy(inp, seed):
    """Same logical K/V under another physical page permutation."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(inp.num_pages, generator=g).to(DEV)
    kc = torch.empty_like(inp.k_cache)
    vc = torch.empty_like(inp.v_cache)
    kc[perm] = inp.k_cache
    vc[perm] = inp.v_cache
    pt = perm[inp.page_table.long()].to(torch.int32)
    return W.DecodeInputs(q=inp.q, k_cache=kc, v_cache=vc, page_table=pt, seq_lens=inp.seq_lens,
                          rel_logits=inp.rel_logits, window=inp.window, scale=inp.scale,
                          max_seq_len=inp.max_seq_len)


@pytest.mark.parametrize("cfg", [(64, 512, 512, 0), (0, 0, 1024, 0), (16, 32, 32, 1)])
def test_page_permutation_bit_exact(ops, cfg):
    P, win, R, tiny = cfg
    if tiny:
        inp = W.make_decode_config("tiny_decode", device=DEV)
    elif win:
        inp = W.make_decode(16, 48, 16, 128, 64, [3000, 511, 64, 1, 700, 8192, 129, 4097] * 2, win,
                            R, device=DEV, seed=3)
    else:
        inp = W.make_decode(6, 48, 8, 128, 64, [20000, 1, 3333, 64, 12345, 9000], 0, R,
                            device=DEV, seed=4)
    out0, lse0 = run(ops, inp)
    for s in range(3):
        out1, lse1 = run(ops, permuted_copy(inp, 50 + s))
        assert np.array_equal(bits(out0), bits(out1))
        assert torch.equal(lse0, lse1)


def _page_of(inp, b, j):
    P = inp.page_size
    return int(inp.page_table[b, j // P]), j % P


@pytest.mark.parametrize("kind", ["local", "global", "tiny"])
def test_one_hot_bias_bit_exact(ops, kind):
    """rel = -1e4 except at distance d*: out must equal the bf16 V row of key
    p - d* bit for bit (pins page-table indexing and the distance)."""
    if kind == "local":
        lens = [1000, 600, 513, 64, 65]
        inp = W.make_decode(5, 48, 16, 128, 64, lens, 512, 512, device=DEV, seed=11)
        dstars = [0, 1, 2, 62, 63, 64, 65, 127, 128, 300, 448, 510, 511]
    elif kind == "global":
        lens = [5000, 3000, 1025]
        inp = W.make_decode(3, 48, 8, 128, 64, lens, 0, 1024, device=DEV, seed=12)
        dstars = [0, 1, 63, 64, 65, 511, 512, 1000, 1022]
    else:
        inp = W.make_decode_config("tiny_decode", device=DEV)
        lens = [37, 100]
        dstars = [0, 1, 15, 16, 17, 31]
    for d in dstars:
        rel = torch.full_like(inp.rel_logits, -1e4)
        rel[:, :, d] = 0.0
        inp2 = W.DecodeInputs(q=inp.q, k_cache=inp.k_cache, v_cache=inp.v_cache,
                              page_table=inp.page_table, seq_lens=inp.seq_lens, rel_logits=rel,
                              window=inp.window, scale=inp.scale, max_seq_len=inp.max_seq_len)
        out, _ = run(ops, inp2)
        G = inp.H_q // inp.H_kv
        for b, L in enumerate(lens):
            if d > L - 1 or (inp.window > 0 and d >= inp.window):
                continue
            page, slot = _page_of(inp, b, L - 1 - d)
            for h in range(inp.H_q):
                want = inp.v_cache[page, slot, h // G]
                assert torch.equal(out[b, h], want), (kind, d, b, h)


@pytest.mark.parametrize("slope", [0.05, 0.3])
def test_rising_bias(ops, slope):
    """A bias that grows toward the most recent keys (rel = -slope * distance)
    raises every row's max along the key walk: by about 4.6 (slope 0.05) or
    28 (slope 0.3) log2 units per 64-key tile, so the exponent base, which is
    re-reduced only when a score passes it by more than 2^8, and the O rescale
    are taken every one to two tiles."""
    import dataclasses
    lens = [700, 1000, 129, 64]
    inp = W.make_decode(4, 48, 8, 128, 64, lens, 0, 1024, device=DEV, seed=21, poison=True)
    d = torch.arange(inp.R, device=DEV, dtype=torch.float32)
    rel = (-slope * d).expand_as(inp.rel_logits).contiguous()
    inp2 = dataclasses.replace(inp, rel_logits=rel)
    for splits in (1, 4):
        out, lse = run(ops, inp2, num_splits=splits)
        ro, rl = oracle_decode(inp2)
        assert_close(out, ro, lse, rl, what=f"slope {slope}, {splits} splits")


def test_single_visible_key_bit_exact(ops):
    lens = [1, 2, 64, 65, 1000]
    inp = W.make_decode(5, 48, 16, 128, 64, lens, 1, 512, device=DEV, seed=13, poison=True,
                        poison_out_of_window=True)
    out, _ = run(ops, inp)
    for b, L in enumerate(lens):
        page, slot = _page_of(inp, b, L - 1)
        for h in range(48):
            assert torch.equal(out[b, h], inp.v_cache[page, slot, h // 3])


def test_nan_outside_window_is_ignored(ops):
    lens = [5000, 600, 513, 2000]
    inp = W.make_decode(4, 48, 16, 128, 64, lens, 512, 512, device=DEV, seed=14, poison=True)
    out0, lse0 = run(ops, inp)
    W.poison_cache(inp.k_cache, inp.v_cache, inp.page_table, inp.seq_lens, inp.meta["used_pages"],
                   window=512, out_of_window=True)
    out1, lse1 = run(ops, inp)
    assert torch.isfinite(out1.float()).all()
    assert np.array_equal(bits(out0), bits(out1)) and torch.equal(lse0, lse1)


# ------------------------------------------------------------------ contract
def test_output_reuse_and_empty_sequences(ops):
    lens = [0, 1, 0, 300]
    inp = W.make_decode(4, 6, 2, 128, 64, lens, 0, 64, device=DEV, seed=15)
    out = torch.full_like(inp.q, float("nan"))
    lse = torch.full((4, 6), 123.0, device=DEV)
    run(ops, inp, out=out, lse=lse)
    ro, rl = oracle_decode(inp)
    assert_close(out, ro, lse, rl, what="reuse")
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.all(lse[0] == -math.inf)


def test_graph_capture_replay(ops):
    """Capture once; change q / seq_lens / page_table / rel in place; replay
    matches an eager call on the new contents (stable-pointer decode)."""
    B, H_q, H_kv, D, P = 8, 48, 8, 128, 64
    lens_a = [5000, 100, 2048, 1, 7000, 64, 333, 4096]
    lens_b = [4000, 7100, 1, 65, 2, 3000, 8000, 129]
    a = W.make_decode(B, H_q, H_kv, D, P, lens_a, 0, 1024, device=DEV, seed=21,
                      max_seq_len=8192, pool_pages=1200)
    b = W.make_decode(B, H_q, H_kv, D, P, lens_b, 0, 1024, device=DEV, seed=22,
                      max_seq_len=8192, pool_pages=1200)
    q = a.q.clone()
    pt = a.page_table.clone()
    sl = a.seq_lens.clone()
    rel = a.rel_logits.clone()
    kc, vc = a.k_cache.clone(), a.v_cache.clone()
    out = torch.empty_like(q)
    lse = torch.empty((B, H_q), device=DEV)
    ws = torch.empty(ops.decode_workspace_bytes(B, H_q, H_kv, D, 0, 8192), dtype=torch.uint8,
                     device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.decode(q, kc, vc, pt, sl, rel, window=0, scale=a.scale, max_seq_len=8192, out=out,
                   lse=lse, workspace=ws)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ops.decode(q, kc, vc, pt, sl, rel, window=0, scale=a.scale, max_seq_len=8192, out=out,
                   lse=lse, workspace=ws)
    for src in (a, b, a):
        q.copy_(src.q)
        pt.copy_(src.page_table)
        sl.copy_(src.seq_lens)
        rel.copy_(src.rel_logits)
        kc.copy_(src.k_cache)
        vc.copy_(src.v_cache)
        g.replay()
        torch.cuda.synchronize()
        eo, el = ops.decode(q, kc, vc, pt, sl, rel, window=0, scale=a.scale, max_seq_len=8192)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(eo)) and torch.equal(lse, el)


def test_bad_page_id_reports_and_reads_zeros(ops):
    inp = W.make_decode(2, 4, 2, 64, 16, [40, 20], 0, 8, device=DEV, seed=30)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pt = inp.page_table.clone()
    pt[0, 1] = inp.num_pages + 5  # out of range: the kernel flags it, TMA zero-fills
    bad = W.DecodeInputs(q=inp.q, k_cache=inp.k_cache, v_cache=inp.v_cache, page_table=pt,
                         seq_lens=inp.seq_lens, rel_logits=inp.rel_logits, window=0,
                         scale=inp.scale, max_seq_len=inp.max_seq_len)
    out, _ = run(ops, bad, device_error=err)
    assert int(err.item()) & 1
    assert torch.isfinite(out.float()).all()
    err.zero_()
    run(ops, inp, device_error=err)
    assert int(err.item()) == 0


def test_seq_longer_than_page_table_row_is_clamped(ops):
    inp = W.make_decode(1, 4, 2, 64, 16, [48], 0, 8, device=DEV, seed=31)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sl = torch.tensor([48 + 16 * 10], dtype=torch.int32, device=DEV)  # beyond stride*P
    long = W.DecodeInputs(q=inp.q, k_cache=inp.k_cache, v_cache=inp.v_cache,
                          page_table=inp.page_table, seq_lens=sl, rel_logits=inp.rel_logits,
                          window=0, scale=inp.scale, max_seq_len=48)
    out, _ = run(ops, long, device_error=err)
    assert int(err.item()) & 2
    assert torch.isfinite(out.float()).all()


def test_workspace_too_small_is_refused(ops):
    from paged_attention_relative_attn_gb300 import _lib
    # 100 keys, full causal: two splits of 64 keys are possible and need workspace
    inp = W.make_decode(2, 4, 2, 64, 16, [37, 100], 0, 32, device=DEV, seed=1)
    out = torch.empty_like(inp.q)
    rc = _lib.inkling_rel_attn_decode(
        inp.q.data_ptr(), inp.k_cache.data_ptr(), inp.v_cache.data_ptr(),
        inp.page_table.data_ptr(), inp.page_table.shape[1], inp.seq_lens.data_ptr(),
        inp.rel_logits.data_ptr(), inp.B, inp.H_q, inp.H_kv, inp.D, inp.page_size, inp.num_pages,
        inp.R, inp.window, inp.scale, inp.max_seq_len, out.data_ptr(), None, None, 0, 2, None,
        torch.cuda.current_stream().cuda_stream)
    assert rc == -3
