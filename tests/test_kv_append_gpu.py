"""KV append through the C ABI against the oracle: the cache after the call
must equal, byte for byte, the oracle's scatter of the new rows (a copy moves
bits, so the bar is bit-exact), and attention over an appended cache must be
bit-identical to attention over the cache that already held those rows."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from oracle.ref import ref_kv_append

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    import paged_attention_relative_attn_gb300 as ira
    from paged_attention_relative_attn_gb300 import build
    build.build()
    return ira


def bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy()


def make_case(q_lens, kv_lens, H_kv, D, P, seed, extra_pages=3):
    g = torch.Generator().manual_seed(seed)
    max_pages = max(W.pages_for(L, P) for L in kv_lens)
    pool = sum(W.pages_for(L, P) for L in kv_lens) + extra_pages
    pt, used = W.build_page_table(kv_lens, P, max_pages, pool, g)
    kc = (torch.randn((pool, P, H_kv, D), generator=g)).to(torch.bfloat16)
    vc = (torch.randn((pool, P, H_kv, D), generator=g)).to(torch.bfloat16)
    # pages no sequence owns hold NaN: a stray write would change them
    owned = torch.zeros(pool, dtype=torch.bool)
    for row, L in zip(pt, kv_lens):
        owned[row[:W.pages_for(L, P)].long()] = True
    kc[~owned] = float("nan")
    vc[~owned] = float("nan")
    T = sum(q_lens)
    k_new = torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens), 0)
    sl = torch.tensor(kv_lens, dtype=torch.int32)
    return dict(k_new=k_new, v_new=v_new, cu=cu, sl=sl, pt=pt.to(torch.int32), kc=kc, vc=vc)


def run_append(ops, c):
    d = {k: v.to(DEV) for k, v in c.items()}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.kv_append(d["k_new"], d["v_new"], d["cu"], d["sl"], d["pt"], d["kc"], d["vc"],
                  device_error=err)
    torch.cuda.synchronize()
    return d["kc"], d["vc"], int(err.item())


def oracle_append(c):
    # bf16 bit patterns as int16: the oracle's scatter moves them unchanged
    kc, vc = ref_kv_append(bits(c["kc"]), bits(c["vc"]), c["pt"].numpy(), c["cu"].numpy(),
                           c["sl"].numpy(), bits(c["k_new"]), bits(c["v_new"]))
    return kc, vc


CASES = [
    # q_lens, kv_lens, H_kv, D, P
    ([1, 1, 1], [9, 64, 200], 2, 64, 16),              # decode: one token each
    ([1, 5, 70], [9, 64, 200], 8, 128, 64),            # mixed chunks, partial / full pages
    ([16, 0, 33], [16, 7, 100], 16, 128, 16),          # a whole first page; an idle sequence
    ([128], [4000], 8, 128, 64),                       # a chunk far into a long sequence
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_append_matches_oracle_bit_exact(ops, case):
    ql, kl, H, D, P = CASES[case]
    c = make_case(ql, kl, H, D, P, seed=40 + case)
    kc, vc, err = run_append(ops, c)
    ek, ev = oracle_append(c)
    assert err == 0
    assert np.array_equal(bits(kc), ek)
    assert np.array_equal(bits(vc), ev)


def test_append_then_decode_is_decode(ops):
    """Decode reads the token it appended: take a decode batch, blank each
    sequence's current token in the cache, append it back, and decode; the
    result must be bit-identical to decoding the untouched cache."""
    inp = W.make_decode(5, 12, 4, 128, 64, [1, 63, 64, 65, 700], 32, 64, device=DEV, seed=9)
    ref_out, ref_lse = ops.decode_inputs(inp)
    B = inp.B
    sl = inp.seq_lens.cpu().tolist()
    pt = inp.page_table.cpu()
    k_new = torch.empty((B, inp.H_kv, inp.D), dtype=torch.bfloat16, device=DEV)
    v_new = torch.empty_like(k_new)
    kc = inp.k_cache.clone()
    vc = inp.v_cache.clone()
    for b, L in enumerate(sl):
        page, slot = int(pt[b, (L - 1) // inp.page_size]), (L - 1) % inp.page_size
        k_new[b] = kc[page, slot]
        v_new[b] = vc[page, slot]
        kc[page, slot] = float("nan")
        vc[page, slot] = float("nan")
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    ops.kv_append(k_new, v_new, cu, inp.seq_lens, inp.page_table, kc, vc)
    out, lse = ops.decode(inp.q, kc, vc, inp.page_table, inp.seq_lens, inp.rel_logits,
                          window=inp.window, scale=inp.scale, max_seq_len=inp.max_seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(ref_out))
    assert torch.equal(lse, ref_lse)


def test_append_then_decode_back_to_back(ops):
    """The same check at a full decode batch, twenty rounds queued on one
    stream with no synchronisation: each round blanks the current tokens'
    rows (a torch kernel), appends them back and decodes.  Decode may start its
    set-up while the append is still running, so this pins that it reads the
    cache only after the append's writes are visible."""
    lens = torch.randint(1024, 8193, (64,), generator=torch.Generator().manual_seed(3)).tolist()
    inp = W.make_decode(64, 48, 16, 128, 64, lens, 512, 512, device=DEV, seed=13)
    ref_out, ref_lse = ops.decode_inputs(inp)
    torch.cuda.synchronize()
    B = inp.B
    pt = inp.page_table.cpu()
    pages = torch.tensor([int(pt[b, (L - 1) // inp.page_size]) for b, L in enumerate(lens)],
                         device=DEV)
    slots = torch.tensor([(L - 1) % inp.page_size for L in lens], device=DEV)
    kc = inp.k_cache.clone()
    vc = inp.v_cache.clone()
    k_new = kc[pages, slots].clone()
    v_new = vc[pages, slots].clone()
    cu = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    outs = []
    for _ in range(20):
        kc[pages, slots] = float("nan")
        vc[pages, slots] = float("nan")
        ops.kv_append(k_new, v_new, cu, inp.seq_lens, inp.page_table, kc, vc)
        out, lse = ops.decode(inp.q, kc, vc, inp.page_table, inp.seq_lens, inp.rel_logits,
                              window=inp.window, scale=inp.scale, max_seq_len=inp.max_seq_len)
        outs.append((out, lse))
    torch.cuda.synchronize()
    for out, lse in outs:
        assert np.array_equal(bits(out), bits(ref_out))
        assert torch.equal(lse, ref_lse)


def test_bad_page_is_reported_and_skipped(ops):
    c = make_case([3, 2], [10, 20], 2, 64, 16, seed=7)
    c["pt"] = c["pt"].clone()
    c["pt"][1, 1] = 10_000  # sequence 1's tokens 18, 19 live in logical page 1
    kc, vc, err = run_append(ops, c)
    assert err & 1  # INKLING_DEVERR_BAD_PAGE
    # sequence 0's tokens are written; nothing else changed
    c0 = dict(c)
    c0["cu"] = torch.tensor([0, 3, 3], dtype=torch.int32)
    c0["k_new"], c0["v_new"] = c["k_new"][:3], c["v_new"][:3]
    ek, ev = oracle_append(c0)
    assert np.array_equal(bits(kc), ek)
    assert np.array_equal(bits(vc), ev)


def test_append_full_size(ops):
    """The bench's append: call 3 of the chunked prefill (4 sequences x 2048
    new tokens at positions 6144..8191, 16 KV heads, pages of 64)."""
    c = make_case([2048] * 4, [8192] * 4, 16, 128, 64, seed=3, extra_pages=0)
    kc, vc, err = run_append(ops, c)
    ek, ev = oracle_append(c)
    assert err == 0
    assert np.array_equal(bits(kc), ek)
    assert np.array_equal(bits(vc), ev)
