"""Pins for the CPU oracle: each check ties ``oracle.ref`` to something other
than itself (brute force, a library routine, a closed form, an invariant that
the mathematics fixes).  ``test_planted_mistakes_are_caught`` plants plausible
mistakes in the oracle's steps and checks that some pin fails for each.

CPU only.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.ref as ref
from oracle.brute import brute_decode, brute_prefill
import workloads as W

F64 = np.float64


def npf(t):
    return t.detach().cpu().float().numpy().astype(F64)


def npi(t):
    return t.detach().cpu().numpy().astype(np.int64)


def decode_args(c):
    return (npf(c.q), npf(c.k_cache), npf(c.v_cache), npi(c.page_table),
            npi(c.seq_lens), npf(c.rel_logits), c.window, c.scale)


def prefill_args(c):
    return (npf(c.q), npi(c.cu_seqlens_q), npf(c.k_cache), npf(c.v_cache),
            npi(c.page_table), npi(c.seq_lens), npf(c.rel_logits), c.window, c.scale)


def scatter_to_pages(K, P, pool_pages, rng):
    """Place contiguous per-sequence rows [L, H, D] into a random paged pool
    (the inverse direction of the oracle's gather, written independently)."""
    B = len(K)
    H, D = K[0].shape[1], K[0].shape[2]
    max_pages = max(1, max((k.shape[0] + P - 1) // P for k in K))
    perm = rng.permutation(pool_pages)
    cache = np.full((pool_pages, P, H, D), np.nan)
    pt = np.zeros((B, max_pages), dtype=np.int64)
    off = 0
    for b, k in enumerate(K):
        L = k.shape[0]
        for lp in range((L + P - 1) // P):
            page = perm[off]
            off += 1
            pt[b, lp] = page
            rows = k[lp * P: (lp + 1) * P]
            cache[page, : rows.shape[0]] = rows
    return cache, pt


# ---------------------------------------------------------------------------
# Pin checks, written as functions of the oracle module so that the planted-
# mistake test can run them against a mutated copy.
# ---------------------------------------------------------------------------

def pin_brute_tiny_decode(R=ref):
    c = W.make_decode_config("tiny_decode")
    out, lse = R.ref_decode(*decode_args(c))
    bo, bl = brute_decode(c.q.float().tolist(), c.k_cache.float().tolist(),
                          c.v_cache.float().tolist(), c.page_table.tolist(),
                          c.seq_lens.tolist(), c.rel_logits.tolist(), c.window,
                          c.scale, c.H_kv)
    np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)
    assert np.isfinite(out).all()


SMALL_CASES = [
    # (B-lengths, H_q, H_kv, D, P, window, R)
    ([5, 1, 17], 3, 1, 8, 4, 0, 4),
    ([9, 12], 4, 2, 4, 4, 3, 8),
    ([33], 6, 2, 4, 8, 0, 6),
    ([0, 7, 2], 2, 2, 4, 4, 5, 5),
    ([20], 2, 1, 4, 16, 20, 3),
]


def pin_brute_small_decode(R=ref):
    for i, (lens, H_q, H_kv, D, P, win, Rr) in enumerate(SMALL_CASES):
        c = W.make_decode(len(lens), H_q, H_kv, D, P, lens, win, Rr, seed=10 + i,
                          pool_pages=sum((L + P - 1) // P for L in lens) + 2,
                          poison=True)
        out, lse = R.ref_decode(*decode_args(c))
        bo, bl = brute_decode(c.q.float().tolist(), c.k_cache.float().tolist(),
                              c.v_cache.float().tolist(), c.page_table.tolist(),
                              c.seq_lens.tolist(), c.rel_logits.tolist(), win,
                              c.scale, H_kv)
        np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def pin_brute_small_prefill(R=ref):
    cases = [([3, 4], [10, 4], 4, 2, 4, 4, 0, 5),
             ([5], [21], 6, 3, 4, 8, 6, 9),
             ([1, 2, 3], [1, 9, 3], 2, 1, 4, 4, 2, 2)]
    for i, (ql, kl, H_q, H_kv, D, P, win, Rr) in enumerate(cases):
        cache = W.make_prefill_cache(kl, H_kv, D, P, seed=20 + i, poison=True,
                                     pool_pages=sum((L + P - 1) // P for L in kl) + 1)
        c = W.make_prefill(cache, ql, kl, H_q, Rr, win, seed=30 + i)
        out, lse = R.ref_prefill(*prefill_args(c))
        bo, bl = brute_prefill(c.q.float().tolist(), c.cu_seqlens_q.tolist(),
                               c.k_cache.float().tolist(), c.v_cache.float().tolist(),
                               c.page_table.tolist(), c.seq_lens.tolist(),
                               c.rel_logits.tolist(), win, c.scale, H_kv)
        np.testing.assert_allclose(out, np.array(bo), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, np.array(bl), rtol=0, atol=1e-12)


def pin_zero_bias_is_sdpa(R=ref):
    """rel_logits = 0 reduces the method to textbook masked GQA attention:
    compare with torch's scaled_dot_product_attention (fp64, CPU, explicit
    boolean mask, its own GQA head expansion) on the contiguous K/V."""
    rng = np.random.default_rng(5)
    for lens, H_q, H_kv, D, P, win, q_len in [([40, 23], 6, 2, 8, 8, 7, 5),
                                               ([64], 4, 4, 16, 16, 0, 64),
                                               ([19, 30, 1], 3, 1, 4, 4, 0, 1)]:
        Ks = [rng.standard_normal((L, H_kv, D)) for L in lens]
        Vs = [rng.standard_normal((L, H_kv, D)) for L in lens]
        pool = sum((L + P - 1) // P for L in lens) + 3
        kc, pt = scatter_to_pages(Ks, P, pool, np.random.default_rng(1))
        vc, _ = scatter_to_pages(Vs, P, pool, np.random.default_rng(1))
        qls = [min(q_len, L) for L in lens]
        T = sum(qls)
        q = rng.standard_normal((T, H_q, D))
        cu = np.concatenate([[0], np.cumsum(qls)])
        rel = np.zeros((T, H_q, 13))
        scale = 1 / math.sqrt(D)
        out, _ = R.ref_prefill(q, cu, kc, vc, pt, np.array(lens), rel, win, scale)
        for b, L in enumerate(lens):
            n = qls[b]
            qq = torch.from_numpy(q[cu[b]:cu[b + 1]]).permute(1, 0, 2)[None]
            kk = torch.from_numpy(Ks[b]).permute(1, 0, 2)[None]
            vv = torch.from_numpy(Vs[b]).permute(1, 0, 2)[None]
            pos = torch.arange(L - n, L)[:, None]
            key = torch.arange(L)[None, :]
            mask = key <= pos
            if win > 0:
                mask &= (pos - key) < win
            o = torch.nn.functional.scaled_dot_product_attention(
                qq, kk, vv, attn_mask=mask, scale=scale, enable_gqa=True)
            np.testing.assert_allclose(out[cu[b]:cu[b + 1]],
                                       o[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def pin_constant_bias_shift(R=ref):
    """A bias constant across distance is a per-row shift: softmax ignores it."""
    c = W.make_decode(3, 4, 2, 8, 8, [50, 9, 30], 0, 16, seed=3)
    a = list(decode_args(c))
    out0, lse0 = R.ref_decode(*a[:5], np.zeros_like(a[5]), *a[6:])
    shift = np.random.default_rng(0).standard_normal(a[5].shape[:2])
    a[5] = np.repeat(shift[:, :, None], a[5].shape[2], axis=2)
    out1, lse1 = R.ref_decode(*a)
    np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1 - shift, lse0, rtol=0, atol=1e-12)


def pin_single_visible_key(R=ref):
    """window = 1: the query sees only its own key, so out = V_p exactly and
    lse = scale*<q, K_p> + rel[..., 0]."""
    c = W.make_decode(2, 4, 2, 8, 4, [13, 1], 1, 6, seed=4, poison=True)
    a = decode_args(c)
    out, lse = R.ref_decode(*a)
    for b, L in enumerate([13, 1]):
        p = L - 1
        page = int(a[3][b, p // 4])
        for h in range(4):
            v = a[2][page, p % 4, h // 2]
            k = a[1][page, p % 4, h // 2]
            assert np.array_equal(out[b, h], v)
            assert lse[b, h] == pytest.approx(c.scale * float(a[0][b, h] @ k) + a[5][b, h, 0],
                                              abs=1e-12)
    # seq_len 1 with no window behaves the same
    c2 = W.make_decode(1, 2, 1, 4, 4, [1], 0, 3, seed=4)
    a2 = decode_args(c2)
    out2, _ = R.ref_decode(*a2)
    page = int(a2[3][0, 0])
    assert np.array_equal(out2[0, 0], a2[2][page, 0, 0])


def pin_one_hot_bias(R=ref):
    """Bias -1e4 everywhere except distance d*: all the weight lands on key
    p - d* (exp(-1e4) underflows to 0 in fp64), so out = V_{p-d*} exactly.
    Pins the page-table indexing and the sign and offset of the distance."""
    c = W.make_decode(2, 4, 2, 8, 4, [23, 11], 0, 32, seed=6)
    a = list(decode_args(c))
    for dstar in [0, 1, 3, 4, 5, 10]:
        rel = np.full_like(a[5], -1e4)
        rel[:, :, dstar] = 0.0
        out, _ = R.ref_decode(*a[:5], rel, *a[6:])
        for b, L in enumerate([23, 11]):
            j = L - 1 - dstar
            page = int(a[3][b, j // 4])
            for h in range(4):
                assert np.array_equal(out[b, h], a[2][page, j % 4, h // 2]), (dstar, b, h)


def pin_window_immunity(R=ref):
    """Keys outside the window (set to NaN, or to other values) do not change
    the result."""
    c = W.make_decode(2, 4, 2, 8, 8, [70, 41], 16, 16, seed=7)
    a = decode_args(c)
    out0, lse0 = R.ref_decode(*a)
    W.poison_cache(c.k_cache, c.v_cache, c.page_table, c.seq_lens,
                   c.meta["used_pages"], window=16, out_of_window=True)
    out1, lse1 = R.ref_decode(*decode_args(c))
    assert np.isfinite(out1).all()
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def pin_page_permutation(R=ref):
    """The same logical K/V under different physical placements gives
    bit-identical results."""
    rng = np.random.default_rng(8)
    lens, H_kv, D, P = [37, 64, 5], 2, 8, 8
    Ks = [rng.standard_normal((L, H_kv, D)) for L in lens]
    Vs = [rng.standard_normal((L, H_kv, D)) for L in lens]
    q = rng.standard_normal((3, 4, D))
    rel = rng.standard_normal((3, 4, 20))
    pool = sum((L + P - 1) // P for L in lens) + 4
    res = []
    for s in range(3):
        kc, pt = scatter_to_pages(Ks, P, pool, np.random.default_rng(100 + s))
        vc, _ = scatter_to_pages(Vs, P, pool, np.random.default_rng(100 + s))
        res.append(R.ref_decode(q, kc, vc, pt, np.array(lens), rel, 30, 0.3))
    for o, l in res[1:]:
        assert np.array_equal(o, res[0][0]) and np.array_equal(l, res[0][1])


def pin_clamp_expansion(R=ref):
    """Distances >= R-1 share the table's last column: a table widened to
    cover every distance by repeating its last column gives the same result."""
    c = W.make_decode(2, 4, 2, 8, 4, [40, 29], 0, 8, seed=9)
    a = list(decode_args(c))
    out0, lse0 = R.ref_decode(*a)
    rel = a[5]
    wide = np.concatenate([rel, np.repeat(rel[:, :, -1:], 40 - rel.shape[2], axis=2)], axis=2)
    out1, lse1 = R.ref_decode(*a[:5], wide, *a[6:])
    np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0, rtol=0, atol=1e-12)
    # and changing only the last column moves the result (the clamp is live)
    rel2 = rel.copy()
    rel2[:, :, -1] += 1.0
    out2, _ = R.ref_decode(*a[:5], rel2, *a[6:])
    assert not np.allclose(out2, out0)


def pin_closed_form(R=ref):
    """Hand-computed example.  One head, D=2, page size 2, pages placed in
    reverse order.  Keys K0=(0,0), K1=(2,0), K2=(1,1); query q=(1,0) at
    position 2; scale 1; R=2 so distance 2 clamps to column 1.
    Scores: s0 = 0 + rel[1] (clamped), s1 = 2 + rel[1], s2 = 1 + rel[0].
    With rel = (0.5, -0.25): s = (-0.25, 1.75, 1.5)."""
    kc = np.zeros((2, 2, 1, 2))
    vc = np.zeros((2, 2, 1, 2))
    # logical page 0 -> physical 1, logical page 1 -> physical 0
    kc[1, 0, 0] = [0, 0]
    kc[1, 1, 0] = [2, 0]
    kc[0, 0, 0] = [1, 1]
    vc[1, 0, 0] = [1, 0]
    vc[1, 1, 0] = [0, 1]
    vc[0, 0, 0] = [3, 3]
    pt = np.array([[1, 0]])
    q = np.array([[[1.0, 0.0]]])
    rel = np.array([[[0.5, -0.25]]])
    s = [-0.25, 1.75, 1.5]
    z = sum(math.exp(x) for x in s)
    w = [math.exp(x) / z for x in s]
    expect = np.array([w[0] * 1 + w[2] * 3, w[1] * 1 + w[2] * 3])
    out, lse = R.ref_decode(q, kc, vc, pt, np.array([3]), rel, 0, 1.0)
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(z), abs=1e-15)
    # window 2 drops key 0: only s1, s2 remain
    out, lse = R.ref_decode(q, kc, vc, pt, np.array([3]), rel, 2, 1.0)
    z2 = math.exp(1.75) + math.exp(1.5)
    np.testing.assert_allclose(out[0, 0], [(math.exp(1.5) * 3) / z2,
                                           (math.exp(1.75) + math.exp(1.5) * 3) / z2],
                               rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(math.log(z2), abs=1e-15)


def pin_decode_is_last_prefill_token(R=ref):
    """Decode is prefill with one query at the end of each sequence."""
    c = W.make_decode(3, 6, 2, 8, 8, [17, 3, 40], 9, 12, seed=11)
    a = decode_args(c)
    o1, l1 = R.ref_decode(*a)
    o2, l2 = R.ref_prefill(a[0], np.arange(4), *a[1:])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_empty_sequence(R=ref):
    c = W.make_decode(2, 2, 1, 4, 4, [0, 5], 0, 4, seed=12)
    out, lse = R.ref_decode(*decode_args(c))
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.all(np.isneginf(lse[0]))
    assert np.isfinite(lse[1]).all()


def pin_kv_append_hand(R=ref):
    """Worked by hand: P = 4, the sequence's pages are [2, 0], 6 tokens in
    total of which the last 3 are appended: positions 3, 4, 5 land in
    (page 2, slot 3), (page 0, slot 0), (page 0, slot 1)."""
    kc = np.zeros((3, 4, 1, 1))
    vc = np.zeros((3, 4, 1, 1))
    k_new = np.array([10.0, 20.0, 30.0]).reshape(3, 1, 1)
    v_new = -k_new
    k2, v2 = R.ref_kv_append(kc, vc, np.array([[2, 0]]), np.array([0, 3]), np.array([6]),
                             k_new, v_new)
    expect = np.zeros((3, 4, 1, 1))
    expect[2, 3] = 10.0
    expect[0, 0] = 20.0
    expect[0, 1] = 30.0
    assert np.array_equal(k2, expect) and np.array_equal(v2, -expect)
    assert np.array_equal(kc, np.zeros_like(kc))  # inputs untouched


def pin_kv_append_readback(R=ref):
    """Append every token of three sequences, in two chunks each, into a
    NaN-poisoned pool laid out by the input generator's page tables; the
    (separately pinned) gather must read back each sequence's values in
    position order, and every slot no token owns must still be NaN."""
    lens = [9, 1, 17]
    P, H, D = 4, 2, 3
    gc = torch.Generator().manual_seed(3)
    max_pages = max(W.pages_for(L, P) for L in lens)
    pool = sum(W.pages_for(L, P) for L in lens) + 2
    pt, _ = W.build_page_table(lens, P, max_pages, pool, gc)
    pt = npi(pt)
    kc = np.full((pool, P, H, D), np.nan)
    vc = np.full((pool, P, H, D), np.nan)
    first = [L // 2 for L in lens]
    for lo_of, hi_of in ((lambda b: 0, lambda b: first[b]), (lambda b: first[b], lambda b: lens[b])):
        q_lens = [hi_of(b) - lo_of(b) for b in range(3)]
        cu = np.concatenate([[0], np.cumsum(q_lens)])
        vals = np.concatenate([1000.0 * b + np.arange(lo_of(b), hi_of(b)) for b in range(3)])
        k_new = np.broadcast_to(vals[:, None, None], (len(vals), H, D)).copy()
        kc, vc = R.ref_kv_append(kc, vc, pt, cu, [hi_of(b) for b in range(3)], k_new, -k_new)
    for b, L in enumerate(lens):
        got = R.gather_sequence(kc, pt[b], L)
        want = np.broadcast_to((1000.0 * b + np.arange(L))[:, None, None], (L, H, D))
        assert np.array_equal(got, want)
        assert np.array_equal(R.gather_sequence(vc, pt[b], L), -want)
    assert int(np.isnan(kc[:, :, 0, 0]).sum()) == pool * P - sum(lens)


def pin_conv_hand(R=ref):
    """Worked by hand, one channel, width 3, taps (0.25, 0.5, 1.0) from the
    oldest input to the current one, state (2, 4):
      chunk (8, 16): y = 0.25*2 + 0.5*4 + 8 = 10.5 and 0.25*4 + 0.5*8 + 16 = 21,
                     new state (8, 16);
      chunk (8):     y = 10.5, new state (4, 8) -- half old state, half new.
    Through the paged append: P = 4, pages [2, 0], 6 tokens of which the last
    2 are new (positions 4, 5 -> page 0 slots 0, 1), state in pool row 1."""
    wgt = np.array([[0.25, 0.5, 1.0]])
    y, st = R.short_conv_chunk(np.array([[8.0], [16.0]]), np.array([[2.0], [4.0]]), wgt)
    assert np.array_equal(y.ravel(), [10.5, 21.0]) and np.array_equal(st.ravel(), [8.0, 16.0])
    y, st = R.short_conv_chunk(np.array([[8.0]]), np.array([[2.0], [4.0]]), wgt)
    assert np.array_equal(y.ravel(), [10.5]) and np.array_equal(st.ravel(), [4.0, 8.0])
    kc = np.zeros((3, 4, 1, 1))
    state = np.zeros((2, 2, 1, 1))
    state[1, :, 0, 0] = [2.0, 4.0]
    k_new = np.array([8.0, 16.0]).reshape(2, 1, 1)
    wk = wgt.reshape(1, 1, 3)
    k2, v2, sk, sv = R.ref_kv_conv_append(kc, kc, np.array([[2, 0]]), np.array([0, 2]),
                                          np.array([6]), k_new, -k_new, wk, 2 * wk,
                                          state, -state, np.array([1]))
    expect = np.zeros((3, 4, 1, 1))
    expect[0, 0], expect[0, 1] = 10.5, 21.0
    assert np.array_equal(k2, expect) and np.array_equal(v2, -2 * expect)
    assert np.array_equal(sk[1, :, 0, 0], [8.0, 16.0]) and np.array_equal(sv[1, :, 0, 0], [-8.0, -16.0])
    assert np.array_equal(sk[0], np.zeros((2, 1, 1)))  # other pool rows untouched


def pin_conv_impulse_response(R=ref):
    """A unit impulse at token 2 (zero state) returns the taps newest first:
    y_{2+k} = weight[:, w-1-k], and zero elsewhere."""
    rng = np.random.default_rng(5)
    C, w, n = 3, 4, 9
    wgt = rng.normal(size=(C, w))
    x = np.zeros((n, C))
    x[2] = 1.0
    y, _ = R.short_conv_chunk(x, np.zeros((w - 1, C)), wgt)
    want = np.zeros((n, C))
    for k in range(w):
        want[2 + k] = wgt[:, w - 1 - k]
    assert np.array_equal(y, want)


def pin_conv_numpy_convolve(R=ref):
    """Each channel equals numpy.convolve of (state, chunk) with the reversed
    taps, 'valid' part; the new state is the last w-1 inputs."""
    rng = np.random.default_rng(6)
    C, w, n = 5, 4, 7
    wgt, st, x = rng.normal(size=(C, w)), rng.normal(size=(w - 1, C)), rng.normal(size=(n, C))
    y, new_st = R.short_conv_chunk(x, st, wgt)
    a = np.concatenate([st, x])
    for c in range(C):
        np.testing.assert_allclose(y[:, c], np.convolve(a[:, c], wgt[c, ::-1], mode="valid"),
                                   rtol=0, atol=1e-12)
    assert np.array_equal(new_st, a[-(w - 1):])


def pin_conv_chunking_invariance(R=ref):
    """Cutting a sequence into chunks (3 + 1 + 6 tokens, the state carried
    between calls) gives exactly the outputs and final state of one call."""
    rng = np.random.default_rng(7)
    C, w, n = 4, 4, 10
    wgt, x = rng.normal(size=(C, w)), rng.normal(size=(n, C))
    y_all, st_all = R.short_conv_chunk(x, np.zeros((w - 1, C)), wgt)
    st, parts, lo = np.zeros((w - 1, C)), [], 0
    for m in (3, 1, 6):
        y, st = R.short_conv_chunk(x[lo:lo + m], st, wgt)
        parts.append(y)
        lo += m
    assert np.array_equal(np.concatenate(parts), y_all) and np.array_equal(st, st_all)


def pin_conv_width1_is_append(R=ref):
    """Width 1 with unit taps is the identity: the convolved append equals
    the (separately pinned) plain append."""
    lens, q_lens, P, H, D = [9, 1, 17], [3, 1, 5], 4, 2, 3
    gc = torch.Generator().manual_seed(8)
    max_pages = max(W.pages_for(L, P) for L in lens)
    pool = sum(W.pages_for(L, P) for L in lens) + 1
    pt, _ = W.build_page_table(lens, P, max_pages, pool, gc)
    pt = npi(pt)
    rng = np.random.default_rng(8)
    kc, vc = rng.normal(size=(pool, P, H, D)), rng.normal(size=(pool, P, H, D))
    T = sum(q_lens)
    k_new, v_new = rng.normal(size=(T, H, D)), rng.normal(size=(T, H, D))
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    ones = np.ones((H, D, 1))
    st = np.zeros((3, 0, H, D))
    k2, v2, _, _ = R.ref_kv_conv_append(kc, vc, pt, cu, lens, k_new, v_new, ones, ones, st, st,
                                        np.array([2, 0, 1]))
    k3, v3 = R.ref_kv_append(kc, vc, pt, cu, lens, k_new, v_new)
    assert np.array_equal(k2, k3) and np.array_equal(v2, v3)


ALL_PINS = [pin_brute_tiny_decode, pin_brute_small_decode, pin_brute_small_prefill,
            pin_zero_bias_is_sdpa, pin_constant_bias_shift, pin_single_visible_key,
            pin_one_hot_bias, pin_window_immunity, pin_page_permutation,
            pin_clamp_expansion, pin_closed_form, pin_decode_is_last_prefill_token,
            pin_empty_sequence, pin_kv_append_hand, pin_kv_append_readback,
            pin_conv_hand, pin_conv_impulse_response, pin_conv_numpy_convolve,
            pin_conv_chunking_invariance, pin_conv_width1_is_append]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin.
# ---------------------------------------------------------------------------

MUTANTS = {
    "gqa_modulo": ("kv_head_of", lambda h, group: h % group),
    "distance_sign": ("distance_index", lambda p, j, R: np.minimum(j - p, R - 1)),
    "clamp_off_by_one": ("distance_index", lambda p, j, R: np.minimum(p - j, R - 2)),
    "window_off_by_one": ("visible", lambda p, j, w: (j <= p) & (((p - j) <= w) if w > 0 else True)),
    "not_causal": ("visible", lambda p, j, w: ((p - j) < w) if w > 0 else np.ones_like(j, bool)),
    "append_position_off_by_one": ("token_positions", lambda cu, sl: (lambda c, s: np.concatenate(
        [[int(s[b]) - int(c[b + 1] - c[b]) + i + 1 for i in range(int(c[b + 1] - c[b]))]
         for b in range(len(s))] + [[]]).astype(np.int64))(np.asarray(cu), np.asarray(sl))),
    "append_slot_transposed": ("cache_slot", lambda row, p, P: (int(row[p // P]), (p // P) % P)),
    "conv_taps_reversed": ("conv_tap_offset", lambda j, w: -j),
    "conv_state_newest_first": ("conv_input", lambda x, st, r: x[r] if r >= 0 else st[-r - 1]),
    "conv_state_off_by_one": ("conv_input",
                              lambda x, st, r: x[r] if r >= 0 else st[max(st.shape[0] + r - 1, 0)]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(ref, attr, fn)
    failures = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ref)
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures > 0, f"mutant {name} passed every pin"


def test_planted_gather_mistake_is_caught(monkeypatch):
    """Reading slot j // P instead of j % P (a transposed index) must fail."""
    def bad_gather(cache, page_row, L):
        P = cache.shape[1]
        out = np.empty((L,) + cache.shape[2:])
        for j in range(L):
            out[j] = cache[int(page_row[j // P]), (j // P) % P]
        return out
    monkeypatch.setattr(ref, "gather_sequence", bad_gather)
    failures = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ref)
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures > 0
