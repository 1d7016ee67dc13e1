"""CPU fp64 oracle for paged attention with a learned relative-position bias.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code,
tables or helpers with the CUDA library.

What it computes (one attention layer of the "Inkling" model as the pages
describe it):

* TensorRT-LLM PR #17062, "Architecture": the model is RoPE-free; position
  enters only through a learned bias added to the scores before the softmax,
  indexed by query token, head and relative distance.  Local layers use a
  sliding window of 512 keys over 16 KV heads, global layers a full causal mask
  over 8 KV heads.
* TensorRT-LLM PR #17062, "Implementation" (``attention_backend/inkling_triton.py``
  row): paged prefill and decode kernels apply the bias as a ``score_mod``; the
  bias tensor ``rel_logits`` has a static shape.
* vLLM PR #51560, "Purpose": attention always runs over the paged KV cache
  (``page_table``).

The pages never write the formula out.  The reading used here (stated once, and
followed literally below):

    K_j     = k_cache[page_table[b, j // P], j % P, h_kv, :]     j = 0 .. L_b - 1
    vis(j)  = j <= p  and  (window <= 0  or  p - j < window)
    s_j     = scale * <q_h, K_j> + rel_logits[t, h, min(p - j, R - 1)]
    out     = sum_{vis} softmax(s)_j V_j ,   lse = log sum_{vis} exp(s_j)

with h_kv = h // (H_q / H_kv) (contiguous GQA groups), p the query's absolute
position, t its packed token index, and a query with no visible key giving
out = 0, lse = -inf.  The bias is added to the already-scaled score, as a
``score_mod`` acts on the scaled score (vLLM PR #51560 discussion: the
FlexAttention fallback carries the bias through ``score_mod``).

Everything is evaluated in float64.  bf16 / fp32 inputs are upcast exactly by
the caller (the arrays given here are already float64 or are cast with
``astype(np.float64)``, which is exact for both).

Each step is a small named function so that tests can plant a mistake in one
of them (monkeypatching) and check that the pins catch it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, textbook SDPA, shift invariance, single key,
one-hot bias, window immunity, page permutation, clamp expansion; for the KV
append a hand-worked example and a read-back through the pinned gather of
values that encode each token's position; for the short convolution a
hand-worked example, the impulse response, ``numpy.convolve``, invariance
under how a sequence is cut into chunks, and width 1 reducing to the plain
append).
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "kv_head_of",
    "distance_index",
    "visible",
    "gather_sequence",
    "attend_sequence",
    "ref_prefill",
    "ref_decode",
    "token_positions",
    "cache_slot",
    "ref_kv_append",
    "conv_tap_offset",
    "conv_input",
    "short_conv_chunk",
    "ref_kv_conv_append",
]


# --------------------------------------------------------------------------
# Small steps of the definition
# --------------------------------------------------------------------------

def kv_head_of(h: int, group: int) -> int:
    """KV head read by query head ``h``: GQA with contiguous groups of ``group``
    query heads per KV head (TensorRT-LLM PR #17062, "Architecture": 48 query
    heads over 16 or 8 KV heads; grouping convention not stated, contiguous
    taken)."""
    return h // group


def distance_index(p, j, R: int):
    """Column of ``rel_logits`` used for a query at position ``p`` and a key at
    position ``j``: the relative distance ``p - j`` clamped to ``R - 1``
    (per (query token, head, relative distance), TensorRT-LLM PR #17062,
    "Architecture"; the clamp bound ``R - 1`` is the last column of the
    static-shape table)."""
    return np.minimum(p - j, R - 1)


def visible(p, j, window: int):
    """Causal mask, plus the sliding window on local layers: key ``j`` is seen
    by the query at ``p`` iff ``j <= p`` and, when ``window > 0``,
    ``p - j < window`` (the window counts the query's own key)."""
    m = j <= p
    if window > 0:
        m = m & ((p - j) < window)
    return m


def gather_sequence(cache: np.ndarray, page_row: np.ndarray, L: int) -> np.ndarray:
    """Logical token rows 0..L-1 of one sequence, read through its page table
    row: token j lives in physical page ``page_row[j // P]`` at slot ``j % P``.

    ``cache`` is [num_pages, P, H_kv, D]; returns float64 [L, H_kv, D].
    """
    P = cache.shape[1]
    out = np.empty((L,) + cache.shape[2:], dtype=np.float64)
    n_pages = (L + P - 1) // P
    for lp in range(n_pages):
        phys = int(page_row[lp])
        n = min(P, L - lp * P)
        out[lp * P: lp * P + n] = cache[phys, :n]
    return out


def attend_sequence(q_rows: np.ndarray, positions: np.ndarray, K: np.ndarray,
                    V: np.ndarray, bias_rows: np.ndarray, window: int,
                    scale: float):
    """Masked, biased softmax attention for the queries of ONE sequence.

    q_rows    [n, H_q, D]  float64
    positions [n]          absolute position of each query
    K, V      [L, H_kv, D] float64, logical order (already gathered)
    bias_rows [n, H_q, R]  float64
    returns out [n, H_q, D], lse [n, H_q]
    """
    n, H_q, D = q_rows.shape
    L, H_kv, _ = K.shape
    R = bias_rows.shape[2]
    group = H_q // H_kv
    out = np.zeros((n, H_q, D), dtype=np.float64)
    lse = np.full((n, H_q), -np.inf, dtype=np.float64)
    j = np.arange(L)
    for i in range(n):
        p = int(positions[i])
        vis = visible(p, j, window)
        if not vis.any():
            continue
        dist = distance_index(p, j[vis], R)
        for h in range(H_q):
            hk = kv_head_of(h, group)
            s = scale * (K[vis, hk, :] @ q_rows[i, h, :]) + bias_rows[i, h, dist]
            m = s.max()
            e = np.exp(s - m)
            z = e.sum()
            out[i, h] = (e @ V[vis, hk, :]) / z
            lse[i, h] = m + math.log(z)
    return out, lse


# --------------------------------------------------------------------------
# Entry points
# --------------------------------------------------------------------------

def ref_prefill(q, cu_seqlens_q, k_cache, v_cache, page_table, seq_lens,
                rel_logits, window: int, scale: float):
    """Chunked / paged prefill (TensorRT-LLM PR #17062, "Implementation":
    paged prefill over the cache).

    Sequence b owns packed query tokens ``cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1``;
    they are the LAST ``q_len_b`` tokens of a sequence whose K/V (prefix and
    this chunk) are already in the cache, so query i sits at position
    ``seq_lens[b] - q_len_b + i``.

    q          [T, H_q, D]              (any float dtype; upcast to float64)
    k/v_cache  [num_pages, P, H_kv, D]
    page_table [B, >= ceil(max L / P)]  int
    seq_lens   [B]                      int, total keys incl. this chunk
    rel_logits [T, H_q, R]
    returns out [T, H_q, D] float64, lse [T, H_q] float64 (natural log)
    """
    q = np.asarray(q, dtype=np.float64)
    rel = np.asarray(rel_logits, dtype=np.float64)
    kc = np.asarray(k_cache)
    vc = np.asarray(v_cache)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    sl = np.asarray(seq_lens, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    T, H_q, D = q.shape
    out = np.zeros((T, H_q, D), dtype=np.float64)
    lse = np.full((T, H_q), -np.inf, dtype=np.float64)
    for b in range(len(sl)):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        n = t1 - t0
        if n == 0:
            continue
        L = int(sl[b])
        if n > L:
            raise ValueError(f"sequence {b}: {n} queries but only {L} keys")
        K = gather_sequence(kc, pt[b], L)
        V = gather_sequence(vc, pt[b], L)
        positions = L - n + np.arange(n)
        o, l = attend_sequence(q[t0:t1], positions, K, V, rel[t0:t1], window, scale)
        out[t0:t1] = o
        lse[t0:t1] = l
    return out, lse


def ref_decode(q, k_cache, v_cache, page_table, seq_lens, rel_logits,
               window: int, scale: float):
    """Decode: one query per sequence, at position ``seq_lens[b] - 1`` (its own
    K/V already written to the cache), packed token index t = b.  A sequence
    with ``seq_lens[b] == 0`` has no visible key: out = 0, lse = -inf.

    q [B, H_q, D], rel_logits [B, H_q, R]; other arguments as ``ref_prefill``.
    """
    q = np.asarray(q, dtype=np.float64)
    rel = np.asarray(rel_logits, dtype=np.float64)
    kc = np.asarray(k_cache)
    vc = np.asarray(v_cache)
    sl = np.asarray(seq_lens, dtype=np.int64)
    pt = np.asarray(page_table, dtype=np.int64)
    B, H_q, D = q.shape
    out = np.zeros((B, H_q, D), dtype=np.float64)
    lse = np.full((B, H_q), -np.inf, dtype=np.float64)
    for b in range(B):
        L = int(sl[b])
        if L == 0:
            continue
        K = gather_sequence(kc, pt[b], L)
        V = gather_sequence(vc, pt[b], L)
        o, l = attend_sequence(q[b:b + 1], np.array([L - 1]), K, V,
                               rel[b:b + 1], window, scale)
        out[b] = o[0]
        lse[b] = l[0]
    return out, lse


# --------------------------------------------------------------------------
# KV append
# --------------------------------------------------------------------------

def token_positions(cu_seqlens_q, seq_lens) -> np.ndarray:
    """Absolute position of every packed token: token i of sequence b (packed
    index ``cu_seqlens_q[b] + i``) is one of the LAST ``q_len_b`` tokens of a
    sequence of ``seq_lens[b]`` tokens, so it sits at ``seq_lens[b] - q_len_b + i``
    (decode: one token per sequence, at ``seq_lens[b] - 1``)."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    sl = np.asarray(seq_lens, dtype=np.int64)
    pos = np.zeros(int(cu[-1]), dtype=np.int64)
    for b in range(len(sl)):
        n = int(cu[b + 1] - cu[b])
        for i in range(n):
            pos[int(cu[b]) + i] = int(sl[b]) - n + i
    return pos


def cache_slot(page_row, p: int, P: int):
    """Physical (page, slot) of logical token ``p`` of a sequence whose page
    table row is ``page_row`` (vLLM PR #51560, "Purpose": attention always runs
    over the paged cache; token p lives in page ``p // P`` of the sequence)."""
    return int(page_row[p // P]), p % P


def ref_kv_append(k_cache, v_cache, page_table, cu_seqlens_q, seq_lens, k_new, v_new):
    """Write the new tokens' K/V into the paged cache (TensorRT-LLM PR #17062,
    commit notes: the attention op itself writes the step's K/V into the cache
    before reading it, hence ``skip_kv_write`` for the backend; vLLM PR #51560,
    "Purpose": the cache is paged through ``page_table``).

    Token t of sequence b at position p (``token_positions``) goes to physical
    page ``page_table[b, p // P]``, slot ``p % P``: all H_kv heads of its K row
    and of its V row.  Every other slot is left as it was.

    k/v_cache [num_pages, P, H_kv, D]; k/v_new [T, H_kv, D].  Returns new
    arrays (the inputs are not modified).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    pt = np.asarray(page_table, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    P = kc.shape[1]
    pos = token_positions(cu_seqlens_q, seq_lens)
    for b in range(len(cu) - 1):
        for t in range(int(cu[b]), int(cu[b + 1])):
            page, slot = cache_slot(pt[b], int(pos[t]), P)
            kc[page, slot] = k_new[t]
            vc[page, slot] = v_new[t]
    return kc, vc


# --------------------------------------------------------------------------
# Causal short convolution on K and V, ahead of the KV append
# --------------------------------------------------------------------------
#
# TensorRT-LLM PR #17062, "Architecture": each layer has four causal short
# convolutions, two of them inside attention (on K and on V), and they carry
# per-request state across decode steps; "pyexecutor" row: that state lives in
# a pool with one row per request.  The pages give neither the width nor the
# layout, so the plainest reading is taken and the width is a parameter:
#
#   * depthwise over the H_kv * D channels of a token's K (resp. V) row, along
#     the token axis, no bias, no activation;
#   * weight[c, j], j = 0 .. w-1: tap j multiplies the input w-1-j tokens back
#     (tap w-1 multiplies the current token):
#         y_t[c] = sum_j weight[c, j] * x_{t-(w-1)+j}[c]
#   * a request's state is its last w-1 inputs (pre-convolution rows), oldest
#     first; a new request's state is zero;
#   * the convolved rows y are what the cache holds (the convolution runs ahead
#     of the append, inside attention).


def conv_tap_offset(j: int, w: int) -> int:
    """Token offset of tap ``j`` of a width-``w`` causal convolution: it
    multiplies the input ``w - 1 - j`` tokens before the current one."""
    return j - (w - 1)


def conv_input(x_chunk: np.ndarray, state: np.ndarray, r: int) -> np.ndarray:
    """Input row at chunk-relative index ``r``: the chunk's own row when
    ``r >= 0``, else row ``(w - 1) + r`` of the request's state (its previous
    ``w - 1`` inputs, oldest first)."""
    return x_chunk[r] if r >= 0 else state[state.shape[0] + r]


def short_conv_chunk(x_chunk, state, weight):
    """One request's new inputs through the causal short convolution.

    x_chunk [n, C] (oldest first), state [w-1, C], weight [C, w].  Returns
    (y [n, C], new_state [w-1, C]): y_i = sum_j weight[:, j] * input at
    i + conv_tap_offset(j, w); the new state is the last w-1 inputs, which
    reach back into the old state when n < w-1.
    """
    x_chunk = np.asarray(x_chunk, dtype=np.float64)
    state = np.asarray(state, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    n, C = x_chunk.shape
    w = weight.shape[1]
    y = np.zeros((n, C))
    for i in range(n):
        for j in range(w):
            y[i] += weight[:, j] * conv_input(x_chunk, state, i + conv_tap_offset(j, w))
    new_state = np.zeros((w - 1, C))
    for j in range(w - 1):
        new_state[j] = conv_input(x_chunk, state, n - (w - 1) + j)
    return y, new_state


def ref_kv_conv_append(k_cache, v_cache, page_table, cu_seqlens_q, seq_lens, k_new, v_new,
                       w_k, w_v, state_k, state_v, state_slots):
    """The short convolutions on K and V of each request's new tokens, then
    the KV append of the convolved rows (see the reading above; the append is
    ``ref_kv_append``'s placement: token t of sequence b at position p goes to
    ``page_table[b, p // P]``, slot ``p % P``).

    k/v_cache [num_pages, P, H_kv, D]; k/v_new [T, H_kv, D]; w_k/w_v
    [H_kv, D, w]; state_k/v [num_slots, w-1, H_kv, D]; state_slots [B], the
    pool row of each sequence (distinct).  Returns new float64 arrays
    (k_cache, v_cache, state_k, state_v); the inputs are not modified.
    """
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    sk = np.array(state_k, dtype=np.float64, copy=True)
    sv = np.array(state_v, dtype=np.float64, copy=True)
    pt = np.asarray(page_table, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    P = kc.shape[1]
    H, D = kc.shape[2], kc.shape[3]
    C = H * D
    w = np.asarray(w_k).shape[2]
    pos = token_positions(cu_seqlens_q, seq_lens)
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        slot = int(state_slots[b])
        outs = []
        for x_new, wt, st in ((k_new, w_k, sk), (v_new, w_v, sv)):
            x = np.asarray(x_new, dtype=np.float64)[t0:t1].reshape(t1 - t0, C)
            y, new_st = short_conv_chunk(x, st[slot].reshape(w - 1, C),
                                         np.asarray(wt, dtype=np.float64).reshape(C, w))
            st[slot] = new_st.reshape(w - 1, H, D)
            outs.append(y.reshape(t1 - t0, H, D))
        for i, t in enumerate(range(t0, t1)):
            page, s = cache_slot(pt[b], int(pos[t]), P)
            kc[page, s] = outs[0][i]
            vc[page, s] = outs[1][i]
    return kc, vc, sk, sv
