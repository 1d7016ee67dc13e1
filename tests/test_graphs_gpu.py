"""CUDA-graph capture and replay of every graph-capturable entry point.

A serving loop captures a call once over stable buffers and, every step,
rewrites those buffers in place (new q, page table, lengths, chunk layout,
state slots) and replays (Support Inkling-NVFP4 model, TensorRT-LLM PR
#17062, "Implementation": the captured forward reads the current batch from
stable buffers).  Each test here captures one call, replays it over several
different contents written in place, and requires the replay to match an
eager call on the same contents bit for bit.  Plain decode has its own
(test_decode_gpu.test_graph_capture_replay)."""

from __future__ import annotations

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ops():
    import paged_attention_relative_attn_gb300 as ira
    from paged_attention_relative_attn_gb300 import build
    build.build()
    return ira


def capture(fn):
    """Warm `fn` up on a side stream, then capture it in a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def same_bits(a, b):
    if a.dtype == torch.bfloat16:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


def test_decode_multi_graph_replay(ops):
    """Multi-token decode over a global layer (split-KV and merge in the
    graph): q, page table, lengths and bias change between replays."""
    q_len, H_q, H_kv, D, P = 4, 48, 8, 128, 64
    # every set holds one 8000-token sequence: the page tables have one width
    lens_sets = [[5000, 100, 2048, 7, 8000, 64], [4000, 8000, 4, 65, 300, 3000],
                 [8000, 7999, 129, 4096, 5, 1000]]
    pool = 8192 // P * 6 + 4
    srcs = []
    for i, lens in enumerate(lens_sets):
        cache = W.make_prefill_cache(lens, H_kv, D, P, device=DEV, seed=400 + i, pool_pages=pool)
        srcs.append(W.make_prefill(cache, [q_len] * len(lens), lens, H_q, 1024, 0, device=DEV,
                                   seed=410 + i, max_seq_len=8192))
    a = srcs[0]
    q, pt, sl, rel = a.q.clone(), a.page_table.clone(), a.seq_lens.clone(), a.rel_logits.clone()
    kc, vc = a.k_cache.clone(), a.v_cache.clone()
    B = sl.shape[0]
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], device=DEV)
    need = ops.decode_multi_workspace_bytes(B, q_len, H_q, H_kv, D, 0, 8192)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)

    def call(o=out, l=lse):
        return ops.decode_multi(q, kc, vc, pt, sl, rel, q_len=q_len, window=0, scale=a.scale,
                                max_seq_len=8192, out=o, lse=l, workspace=ws)

    g = capture(call)
    for src in srcs + [srcs[1]]:
        for dst, s in ((q, src.q), (pt, src.page_table), (sl, src.seq_lens), (rel, src.rel_logits),
                       (kc, src.k_cache), (vc, src.v_cache)):
            dst.copy_(s)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        eo, el = call(torch.empty_like(out), torch.empty_like(lse))
        torch.cuda.synchronize()
        assert same_bits(out, eo) and same_bits(lse, el)


def test_prefill_graph_replay(ops):
    """Chunked prefill over a local layer: the chunk layout (cu_seqlens_q),
    the lengths, q and the bias change between replays; T and max_q_len (host
    scalars of the captured call) stay."""
    H_q, H_kv, D, P, W_, R = 12, 4, 128, 64, 512, 512
    T, max_q = 700, 400
    totals = [3000, 2500, 900]
    cache = W.make_prefill_cache(totals, H_kv, D, P, device=DEV, seed=420)
    layouts = [([400, 200, 100], [1400, 2500, 900]),
               ([1, 399, 300], [3000, 1000, 300]),
               ([300, 0, 400], [700, 2500, 400])]
    srcs = []
    for i, (ql, kl) in enumerate(layouts):
        assert sum(ql) == T and max(ql) <= max_q
        srcs.append(W.make_prefill(cache, ql, kl, H_q, R, W_, device=DEV, seed=430 + i,
                                   max_seq_len=3000))
    a = srcs[0]
    q, cu, sl, rel = a.q.clone(), a.cu_seqlens_q.clone(), a.seq_lens.clone(), a.rel_logits.clone()
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], device=DEV)

    def call(o=out, l=lse):
        return ops.prefill(q, cu, a.k_cache, a.v_cache, a.page_table, sl, rel, window=W_,
                           scale=a.scale, max_seq_len=3000, max_q_len=max_q, out=o, lse=l)

    g = capture(call)
    for src in srcs + [srcs[0]]:
        for dst, s in ((q, src.q), (cu, src.cu_seqlens_q), (sl, src.seq_lens),
                       (rel, src.rel_logits)):
            dst.copy_(s)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        eo, el = call(torch.empty_like(out), torch.empty_like(lse))
        torch.cuda.synchronize()
        assert same_bits(out, eo) and same_bits(lse, el)


def _append_case(seed, T=600):
    H_kv, D, P = 8, 128, 64
    g = torch.Generator().manual_seed(seed)
    totals = [2000, 1500, 700]
    pool = sum(W.pages_for(L, P) for L in totals) + 2
    pt, _ = W.build_page_table(totals, P, W.pages_for(2000, P), pool, g)
    kc = torch.randn((pool, P, H_kv, D), generator=g).to(torch.bfloat16).to(DEV)
    vc = torch.randn((pool, P, H_kv, D), generator=g).to(torch.bfloat16).to(DEV)
    return pt.to(torch.int32).to(DEV), kc, vc, H_kv, D


APPEND_LAYOUTS = [([300, 200, 100], [1300, 1200, 700]),
                  ([1, 299, 300], [2000, 700, 300]),
                  ([600, 0, 0], [1900, 1500, 700])]


def test_kv_append_graph_replay(ops):
    """KV append: the new rows, the chunk layout and the lengths change
    between replays; the cache written by the replay equals the cache
    written by an eager call from the same starting contents."""
    pt, kc0, vc0, H_kv, D = _append_case(440)
    T = 600
    g_ = torch.Generator(device=DEV).manual_seed(441)
    k_new = torch.empty((T, H_kv, D), dtype=torch.bfloat16, device=DEV)
    v_new = torch.empty_like(k_new)
    cu = torch.zeros(4, dtype=torch.int32, device=DEV)
    sl = torch.zeros(3, dtype=torch.int32, device=DEV)
    kc, vc = kc0.clone(), vc0.clone()
    graph = capture(lambda: ops.kv_append(k_new, v_new, cu, sl, pt, kc, vc))
    for ql, kl in APPEND_LAYOUTS + [APPEND_LAYOUTS[0]]:
        k_new.copy_(torch.randn((T, H_kv, D), generator=g_, device=DEV).to(torch.bfloat16))
        v_new.copy_(torch.randn((T, H_kv, D), generator=g_, device=DEV).to(torch.bfloat16))
        cu.copy_(torch.tensor([0] + list(torch.tensor(ql).cumsum(0)), dtype=torch.int32))
        sl.copy_(torch.tensor(kl, dtype=torch.int32))
        kc.copy_(kc0)
        vc.copy_(vc0)
        graph.replay()
        ek, ev = kc0.clone(), vc0.clone()
        ops.kv_append(k_new, v_new, cu, sl, pt, ek, ev)
        torch.cuda.synchronize()
        assert same_bits(kc, ek) and same_bits(vc, ev)
        assert not same_bits(kc, kc0)  # the call wrote something


def test_kv_conv_append_graph_replay(ops):
    """Short convolution + append: new rows, chunk layout, lengths and the
    state slots change between replays; cache and state pool written by the
    replay equal those written by an eager call from the same contents."""
    pt, kc0, vc0, H_kv, D = _append_case(450)
    T, width, n_slots = 600, 4, 6
    g_ = torch.Generator(device=DEV).manual_seed(451)
    k_new = torch.empty((T, H_kv, D), dtype=torch.bfloat16, device=DEV)
    v_new = torch.empty_like(k_new)
    cu = torch.zeros(4, dtype=torch.int32, device=DEV)
    sl = torch.zeros(3, dtype=torch.int32, device=DEV)
    slots = torch.zeros(3, dtype=torch.int32, device=DEV)
    w_k = 0.5 * torch.randn((H_kv, D, width), generator=g_, device=DEV)
    w_v = 0.5 * torch.randn((H_kv, D, width), generator=g_, device=DEV)
    s_k0 = torch.randn((n_slots, width - 1, H_kv, D), generator=g_, device=DEV).to(torch.bfloat16)
    s_v0 = torch.randn((n_slots, width - 1, H_kv, D), generator=g_, device=DEV).to(torch.bfloat16)
    kc, vc, s_k, s_v = kc0.clone(), vc0.clone(), s_k0.clone(), s_v0.clone()
    graph = capture(lambda: ops.kv_conv_append(k_new, v_new, cu, sl, pt, kc, vc, w_k, w_v, s_k,
                                               s_v, slots, max_q_len=600))
    slot_sets = [[0, 1, 2], [5, 3, 1], [4, 0, 2]]
    for (ql, kl), sset in zip(APPEND_LAYOUTS + [APPEND_LAYOUTS[1]], slot_sets + [slot_sets[0]]):
        k_new.copy_(torch.randn((T, H_kv, D), generator=g_, device=DEV).to(torch.bfloat16))
        v_new.copy_(torch.randn((T, H_kv, D), generator=g_, device=DEV).to(torch.bfloat16))
        cu.copy_(torch.tensor([0] + list(torch.tensor(ql).cumsum(0)), dtype=torch.int32))
        sl.copy_(torch.tensor(kl, dtype=torch.int32))
        slots.copy_(torch.tensor(sset, dtype=torch.int32))
        for dst, src in ((kc, kc0), (vc, vc0), (s_k, s_k0), (s_v, s_v0)):
            dst.copy_(src)
        graph.replay()
        ek, ev, esk, esv = kc0.clone(), vc0.clone(), s_k0.clone(), s_v0.clone()
        ops.kv_conv_append(k_new, v_new, cu, sl, pt, ek, ev, w_k, w_v, esk, esv, slots,
                           max_q_len=600)
        torch.cuda.synchronize()
        assert same_bits(kc, ek) and same_bits(vc, ev)
        assert same_bits(s_k, esk) and same_bits(s_v, esv)
        assert not same_bits(s_k, s_k0)  # the state rows moved on
