"""The short convolution on K and V ahead of the KV append, through the C ABI,
against the oracle.  The state rows are raw copies of inputs (bit-exact); the
convolved cache rows are fp32 sums rounded to bf16, compared with the fp64
oracle within one bf16 rounding plus the fp32 accumulation error; every cache
byte the call must not write is checked bit for bit (NaN poison)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from oracle.ref import ref_kv_append, ref_kv_conv_append, short_conv_chunk

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


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def make_case(q_lens, kv_lens, H_kv, D, P, width, seed, num_slots=None):
    g = torch.Generator().manual_seed(seed)
    B = len(q_lens)
    max_pages = max(W.pages_for(L, P) for L in kv_lens)
    pool = sum(W.pages_for(L, P) for L in kv_lens) + 2
    pt, _ = W.build_page_table(kv_lens, P, max_pages, pool, g)
    kc = torch.randn((pool, P, H_kv, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((pool, P, H_kv, D), generator=g).to(torch.bfloat16)
    owned = torch.zeros(pool, dtype=torch.bool)
    for row, L in zip(pt, kv_lens):
        owned[row[:W.pages_for(L, P)].long()] = True
    kc[~owned] = float("nan")  # a stray write would change these
    vc[~owned] = float("nan")
    T = sum(q_lens)
    num_slots = num_slots or B + 3
    slots = torch.randperm(num_slots, generator=g)[:B].to(torch.int32)
    c = dict(
        k_new=torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16),
        v_new=torch.randn((T, H_kv, D), generator=g).to(torch.bfloat16),
        cu=torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32),
        sl=torch.tensor(kv_lens, dtype=torch.int32), pt=pt.to(torch.int32), kc=kc, vc=vc,
        w_k=(0.5 * torch.randn((H_kv, D, width), generator=g)).float(),
        w_v=(0.5 * torch.randn((H_kv, D, width), generator=g)).float(),
        s_k=torch.randn((num_slots, width - 1, H_kv, D), generator=g).to(torch.bfloat16),
        s_v=torch.randn((num_slots, width - 1, H_kv, D), generator=g).to(torch.bfloat16),
        slots=slots, max_q_len=max(q_lens))
    return c


def run(ops, c, **over):
    d = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in c.items()}
    d.update(over)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ops.kv_conv_append(d["k_new"], d["v_new"], d["cu"], d["sl"], d["pt"], d["kc"], d["vc"],
                       d["w_k"], d["w_v"], d["s_k"], d["s_v"], d["slots"],
                       max_q_len=d["max_q_len"], device_error=err)
    torch.cuda.synchronize()
    return d, int(err.item())


def oracle(c):
    return ref_kv_conv_append(f64(c["kc"]), f64(c["vc"]), c["pt"].numpy(), c["cu"].numpy(),
                              c["sl"].numpy(), f64(c["k_new"]), f64(c["v_new"]),
                              c["w_k"].numpy(), c["w_v"].numpy(), f64(c["s_k"]), f64(c["s_v"]),
                              c["slots"].numpy())


def magnitude(c):
    """sum_j |w_j| |x_j| of every output (the scale of the fp32 accumulation
    error), by the same oracle on absolute values."""
    a = {k: (v.abs() if torch.is_tensor(v) and v.is_floating_point() else v) for k, v in c.items()}
    mk, mv, _, _ = oracle(a)
    return mk, mv


def assert_conv_close(got, want, mag, what):
    g = f64(got)
    finite = ~np.isnan(want)
    assert np.array_equal(np.isnan(g), ~finite), f"{what}: NaN pattern differs"
    tol = 2.0 ** -8 * np.abs(want[finite]) + 2.0 ** -20 * mag[finite] + 1e-30
    err = np.abs(g[finite] - want[finite])
    assert np.all(err <= tol), f"{what}: max excess {float(np.max(err - tol)):.3g}"


CASES = [
    # q_lens, kv_lens, H_kv, D, P, width
    ([1, 1, 1], [9, 64, 200], 2, 64, 16, 4),           # decode steps
    ([1, 5, 70], [9, 64, 200], 8, 128, 64, 4),         # mixed chunks; a token shorter than the window
    ([2, 1, 150], [40, 7, 400], 4, 128, 16, 8),        # chunks shorter than the window; several segments
    ([16, 0, 33], [16, 7, 100], 16, 128, 64, 3),       # a whole first page; an idle sequence
    ([3, 65, 1], [3, 65, 20], 2, 64, 16, 2),           # a request's first tokens
    ([128], [4000], 8, 128, 64, 4),                    # a chunk far into a long sequence
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_conv_append_matches_oracle(ops, case):
    ql, kl, H, D, P, w = CASES[case]
    c = make_case(ql, kl, H, D, P, w, seed=60 + case)
    d, err = run(ops, c)
    assert err == 0
    ek, ev, esk, esv = oracle(c)
    mk, mv = magnitude(c)
    assert_conv_close(d["kc"], ek, np.nan_to_num(mk), "k_cache")
    assert_conv_close(d["vc"], ev, np.nan_to_num(mv), "v_cache")
    # state rows are raw inputs: bit-exact, and only the sequences' rows change
    assert np.array_equal(f64(d["s_k"]), esk) and np.array_equal(f64(d["s_v"]), esv)


def test_untouched_bytes_bit_exact(ops):
    """Cache slots no new token owns, and pool rows no sequence uses, keep
    their exact bits."""
    c = make_case([2, 1, 150], [40, 7, 400], 4, 128, 16, 8, seed=70)
    d, err = run(ops, c)
    assert err == 0
    ek, _, _, _ = oracle(c)
    before = bits(c["kc"])
    after = bits(d["kc"])
    old = f64(c["kc"])
    written = (ek != old) & ~(np.isnan(ek) & np.isnan(old))  # NaN == NaN: not written
    assert np.isnan(old[~written]).any()  # the poisoned pages are among the checked bytes
    assert np.array_equal(after[~written], before[~written])
    used = set(c["slots"].tolist())
    for s in range(c["s_k"].shape[0]):
        if s not in used:
            assert np.array_equal(bits(d["s_k"][s]), bits(c["s_k"][s]))


def test_chunking_is_bit_exact(ops):
    """One sequence's 100 new tokens in one call, or in calls of 3, 1, 60 and
    36 tokens with the state carried: the same cache rows and state, bit for
    bit (each output sums the same inputs in the same order)."""
    whole = make_case([100], [300], 8, 128, 64, 4, seed=71)
    d1, err = run(ops, whole)
    assert err == 0
    kc, vc, sk, sv = (whole[k].clone().to(DEV) for k in ("kc", "vc", "s_k", "s_v"))
    done = 200  # tokens already in the cache before the 100 new ones
    lo = 0
    for n in (3, 1, 60, 36):
        part = dict(whole)
        part.update(k_new=whole["k_new"][lo:lo + n], v_new=whole["v_new"][lo:lo + n],
                    cu=torch.tensor([0, n], dtype=torch.int32),
                    sl=torch.tensor([done + lo + n], dtype=torch.int32), max_q_len=n,
                    kc=kc, vc=vc, s_k=sk, s_v=sv)
        _, err = run(ops, part)
        assert err == 0
        lo += n
    assert np.array_equal(bits(kc), bits(d1["kc"])) and np.array_equal(bits(vc), bits(d1["vc"]))
    assert np.array_equal(bits(sk), bits(d1["s_k"])) and np.array_equal(bits(sv), bits(d1["s_v"]))


def test_width_one_is_append_bit_exact(ops):
    c = make_case([1, 5, 70], [9, 64, 200], 8, 128, 64, 1, seed=72)
    c["w_k"] = torch.ones_like(c["w_k"])
    c["w_v"] = torch.ones_like(c["w_v"])
    d, err = run(ops, c, s_k=None, s_v=None, slots=None)
    assert err == 0
    ek, ev = ref_kv_append(bits(c["kc"]), bits(c["vc"]), c["pt"].numpy(), c["cu"].numpy(),
                           c["sl"].numpy(), bits(c["k_new"]), bits(c["v_new"]))
    assert np.array_equal(bits(d["kc"]), ek) and np.array_equal(bits(d["vc"]), ev)


def test_bad_slot_is_reported_and_skipped(ops):
    c = make_case([3, 2], [10, 20], 2, 64, 16, 4, seed=73, num_slots=4)
    c["slots"] = torch.tensor([1, 9], dtype=torch.int32)  # 9 is outside the pool
    d, err = run(ops, c)
    assert err & 16  # INKLING_DEVERR_BAD_SLOT
    # sequence 0 is written and its state advanced; sequence 1 changes nothing
    c0 = dict(c)
    c0.update(cu=torch.tensor([0, 3, 3], dtype=torch.int32),
              k_new=c["k_new"][:3], v_new=c["v_new"][:3], slots=torch.tensor([1, 2], dtype=torch.int32))
    ek, _, esk, _ = oracle(c0)
    mk, _ = magnitude(c0)
    assert_conv_close(d["kc"], ek, np.nan_to_num(mk), "k_cache")
    assert np.array_equal(f64(d["s_k"]), esk)


def test_full_size_chunk(ops):
    """The bench's size: one chunked-prefill call (4 sequences x 2048 new
    tokens at positions 6144..8191, 16 KV heads, D = 128, pages of 64), width
    4; the oracle convolution per sequence, read back from the paged cache."""
    c = make_case([2048] * 4, [8192] * 4, 16, 128, 64, 4, seed=74)
    d, err = run(ops, c)
    assert err == 0
    kc = d["kc"]
    C = 16 * 128
    for b in range(4):
        t0 = 2048 * b
        x = f64(c["k_new"][t0:t0 + 2048]).reshape(2048, C)
        st = f64(c["s_k"][int(c["slots"][b])]).reshape(3, C)
        wk = c["w_k"].numpy().astype(np.float64).reshape(C, 4)
        y, new_st = short_conv_chunk(x, st, wk)
        mag, _ = short_conv_chunk(np.abs(x), np.abs(st), np.abs(wk))
        pos = 8192 - 2048 + np.arange(2048)
        pages = c["pt"][b, torch.from_numpy(pos // 64)].long()
        got = kc[pages.to(DEV), torch.from_numpy(pos % 64).to(DEV)].reshape(2048, C)
        assert_conv_close(got, y, mag, f"sequence {b}")
        assert np.array_equal(f64(d["s_k"][int(c["slots"][b])]).reshape(3, C), new_st)
