"""Scalar brute-force evaluation of the same definition as ``oracle.ref``.

TEST INFRASTRUCTURE ONLY (see ``oracle/ref.py`` for who may call it).

It exists to pin ``oracle.ref`` on tiny inputs: plain Python loops over
sequences, heads, queries and keys, ``math.exp`` / ``math.log``, the page table
read afresh for every key, no NumPy arithmetic, no masking arrays and no
vectorised gather.  Inputs are nested Python lists (or anything indexable that
yields Python floats / ints).

Definition followed (Support Inkling-NVFP4 model, TensorRT-LLM PR #17062,
"Architecture": bias per (query token, head, relative distance) added before
the softmax; RoPE-free): for a query at position p in sequence b, head h,

    s_j = scale * sum_d q[h][d] * K_j[d]  +  rel[h][min(p - j, R - 1)]
    over keys j with 0 <= p - j (and p - j < window when window > 0)
"""

from __future__ import annotations

import math


def brute_query(q_row, p, L, b, k_cache, v_cache, page_table, bias_row,
                window, scale, H_kv):
    """One query token, all heads.  Returns (out[h][d], lse[h]) as lists."""
    H_q = len(q_row)
    D = len(q_row[0])
    P = len(k_cache[0])
    R = len(bias_row[0])
    group = H_q // H_kv
    outs, lses = [], []
    for h in range(H_q):
        hk = h // group
        scores, values = [], []
        for j in range(L):
            if j > p:
                continue
            if window > 0 and p - j >= window:
                continue
            page = int(page_table[b][j // P])
            slot = j % P
            krow = k_cache[page][slot][hk]
            dot = 0.0
            for d in range(D):
                dot += float(q_row[h][d]) * float(krow[d])
            dist = p - j
            if dist > R - 1:
                dist = R - 1
            scores.append(scale * dot + float(bias_row[h][dist]))
            values.append(v_cache[page][slot][hk])
        if not scores:
            outs.append([0.0] * D)
            lses.append(-math.inf)
            continue
        m = max(scores)
        w = [math.exp(s - m) for s in scores]
        z = sum(w)
        o = [0.0] * D
        for wj, vrow in zip(w, values):
            for d in range(D):
                o[d] += wj * float(vrow[d])
        outs.append([x / z for x in o])
        lses.append(m + math.log(z))
    return outs, lses


def brute_decode(q, k_cache, v_cache, page_table, seq_lens, rel_logits,
                 window, scale, H_kv):
    """Decode: query b at position seq_lens[b] - 1."""
    outs, lses = [], []
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        o, l = brute_query(q[b], L - 1, L, b, k_cache, v_cache, page_table,
                           rel_logits[b], window, scale, H_kv)
        outs.append(o)
        lses.append(l)
    return outs, lses


def brute_prefill(q, cu_seqlens_q, k_cache, v_cache, page_table, seq_lens,
                  rel_logits, window, scale, H_kv):
    """Prefill: query i of sequence b at position seq_lens[b] - q_len_b + i."""
    outs, lses = [], []
    for b in range(len(seq_lens)):
        t0, t1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        L = int(seq_lens[b])
        n = t1 - t0
        for i in range(n):
            p = L - n + i
            o, l = brute_query(q[t0 + i], p, L, b, k_cache, v_cache, page_table,
                               rel_logits[t0 + i], window, scale, H_kv)
            outs.append(o)
            lses.append(l)
    return outs, lses
