"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only DRAWS inputs (shapes, value distributions, sequence lengths,
page shuffles, NaN poison).  It holds none of the attention arithmetic, so the
CUDA path and the CPU oracle stay independent of each other: both receive the
same tensors from here.

Workloads (all synthetic; no dataset or weights exist for this path):

* ``tiny_decode``     B=2, H_q=4, H_kv=2, D=64, page 16, lengths {37, 100},
                      window 32, R=32, 16-page pool (10 used, 6 NaN-poisoned).
* ``local_decode``    B=64, H_q=48, H_kv=16, D=128, page 64, lengths uniform in
                      [1024, 8192], window 512, R=512.
* ``global_decode``   B=32, H_q=48, H_kv=8, D=128, page 64, lengths uniform in
                      [4096, 32768], full causal, R=1024, split-KV.
* ``chunked_prefill`` 4 sequences x 8192 tokens in 2048-token chunks against the
                      cached prefix, H_q=48, H_kv=16, D=128, window 512, R=512.
* ``decode_66_layers`` 55 local + 11 global layers (layer l global iff l % 6 == 5),
                      B=128, lengths lognormal with mean 2048 (sigma 0.5),
                      clipped to [1, 8192].

Value recipe: q, K, V ~ N(0, 1) rounded to bf16; rel_logits ~ N(0, 0.5^2) in
fp32; scale = 1/sqrt(D); physical pages are a random permutation of the pool,
the pool holding exactly the pages the sequences use unless stated.  Sequence
structure (lengths, permutation) is drawn on a CPU generator so it is the same
on every device; bulk values are drawn on the target device's generator.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

BF16 = torch.bfloat16


# ---------------------------------------------------------------------------
# Containers
# ---------------------------------------------------------------------------

@dataclass
class DecodeInputs:
    q: torch.Tensor            # [B, H_q, D] bf16
    k_cache: torch.Tensor      # [num_pages, P, H_kv, D] bf16
    v_cache: torch.Tensor      # [num_pages, P, H_kv, D] bf16
    page_table: torch.Tensor   # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32 (includes the current token)
    rel_logits: torch.Tensor   # [B, H_q, R] fp32
    window: int                # <= 0: full causal
    scale: float
    max_seq_len: int           # host-side bound on seq_lens
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def H_q(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def H_kv(self):
        return self.k_cache.shape[2]

    @property
    def page_size(self):
        return self.k_cache.shape[1]

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def R(self):
        return self.rel_logits.shape[2]


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H_q, D] bf16
    cu_seqlens_q: torch.Tensor # [B+1] int32
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor   # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32, total keys incl. this chunk
    rel_logits: torch.Tensor   # [T, H_q, R] fp32
    window: int
    scale: float
    max_seq_len: int
    max_q_len: int
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.seq_lens.shape[0]

    @property
    def T(self):
        return self.q.shape[0]

    @property
    def H_q(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def H_kv(self):
        return self.k_cache.shape[2]

    @property
    def page_size(self):
        return self.k_cache.shape[1]

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def R(self):
        return self.rel_logits.shape[2]


# ---------------------------------------------------------------------------
# Draw helpers
# ---------------------------------------------------------------------------

def _cpu_gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _dev_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, gen, device, dtype, std=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def _fill_randn_bf16(t: torch.Tensor, gen):
    """Fill a (possibly huge) bf16 tensor with N(0,1) in slices to bound the
    fp32 temporary."""
    flat = t.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        e = min(flat.numel(), s + step)
        flat[s:e] = torch.randn(e - s, generator=gen, device=t.device,
                                dtype=torch.float32).to(BF16)


def pages_for(L: int, P: int) -> int:
    return (L + P - 1) // P


def build_page_table(seq_lens, P, max_pages, pool_pages, gen_cpu):
    """Random physical placement: the pages the sequences use are taken, in
    order, from a random permutation of the pool.  Returns (page_table int32
    [B, max_pages] with unused entries 0, list of used page ids)."""
    perm = torch.randperm(pool_pages, generator=gen_cpu)
    B = len(seq_lens)
    pt = torch.zeros((B, max_pages), dtype=torch.int32)
    used = []
    off = 0
    for b, L in enumerate(seq_lens):
        n = pages_for(int(L), P)
        ids = perm[off: off + n]
        pt[b, :n] = ids.to(torch.int32)
        used.extend(int(x) for x in ids)
        off += n
    if off > pool_pages:
        raise ValueError("pool too small")
    return pt, used


def poison_cache(k_cache, v_cache, page_table, seq_lens, used_pages, window=0,
                 out_of_window=False):
    """Write NaN where no visible key lives: pool pages no sequence uses, the
    slots of each sequence's last page past its length and, optionally, every
    key outside the decode query's window.  Correct code never lets these
    values reach an output."""
    P = k_cache.shape[1]
    num_pages = k_cache.shape[0]
    nan = float("nan")
    used = set(used_pages)
    unused = [p for p in range(num_pages) if p not in used]
    if unused:
        idx = torch.tensor(unused, device=k_cache.device, dtype=torch.long)
        k_cache.index_fill_(0, idx, nan)
        v_cache.index_fill_(0, idx, nan)
    pt = page_table.cpu()
    for b, L in enumerate(seq_lens.cpu().tolist()):
        L = int(L)
        n = pages_for(L, P)
        if n and L % P:
            last = int(pt[b, n - 1])
            k_cache[last, L % P:] = nan
            v_cache[last, L % P:] = nan
        if out_of_window and window > 0 and L > window:
            lo = L - window  # first visible key of the decode query at L-1
            for j0 in range(0, lo, P):
                page = int(pt[b, j0 // P])
                e = min(P, lo - j0)
                k_cache[page, :e] = nan
                v_cache[page, :e] = nan


# ---------------------------------------------------------------------------
# Decode
# ---------------------------------------------------------------------------

DECODE_CONFIGS = {
    "tiny_decode": dict(B=2, H_q=4, H_kv=2, D=64, P=16, seq_lens=[37, 100],
                        window=32, R=32, pool_pages=16, max_seq_len=100),
    "local_decode": dict(B=64, H_q=48, H_kv=16, D=128, P=64,
                         len_range=(1024, 8192), window=512, R=512),
    "global_decode": dict(B=32, H_q=48, H_kv=8, D=128, P=64,
                          len_range=(4096, 32768), window=0, R=1024),
}


def make_decode(B, H_q, H_kv, D, P, seq_lens, window, R, *, device="cpu",
                seed=0, pool_pages=None, max_seq_len=None, poison=False,
                poison_out_of_window=False, name="", rel_std=0.5, q_std=1.0):
    """Draw one decode batch.  ``seq_lens`` is a list of ints (0 allowed)."""
    gc = _cpu_gen(seed)
    seq_lens = [int(x) for x in seq_lens]
    if max_seq_len is None:
        max_seq_len = max(seq_lens + [1])
    max_pages = max(1, pages_for(max_seq_len, P))
    need = sum(pages_for(L, P) for L in seq_lens)
    if pool_pages is None:
        pool_pages = max(need, 1)
    pt, used = build_page_table(seq_lens, P, max_pages, pool_pages, gc)
    gd = _dev_gen(seed + 1, device)
    q = _randn((B, H_q, D), gd, device, BF16, std=q_std)
    k_cache = torch.empty((pool_pages, P, H_kv, D), dtype=BF16, device=device)
    v_cache = torch.empty_like(k_cache)
    _fill_randn_bf16(k_cache, gd)
    _fill_randn_bf16(v_cache, gd)
    rel = _randn((B, H_q, R), gd, device, torch.float32, std=rel_std)
    sl = torch.tensor(seq_lens, dtype=torch.int32)
    if poison:
        poison_cache(k_cache, v_cache, pt, sl, used, window, poison_out_of_window)
    return DecodeInputs(q=q, k_cache=k_cache, v_cache=v_cache,
                        page_table=pt.to(device), seq_lens=sl.to(device),
                        rel_logits=rel, window=window, scale=1.0 / math.sqrt(D),
                        max_seq_len=max_seq_len, name=name,
                        meta=dict(used_pages=used))


def draw_uniform_lengths(B, lo, hi, seed):
    """Sequence lengths uniform on the integers lo..hi inclusive."""
    g = _cpu_gen(seed + 1000)
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def make_decode_config(name, *, device="cpu", seed=0, poison=None, batch=None):
    """One of the named decode workloads.  ``batch`` keeps only the first
    ``batch`` sequences (same lengths / placement draw as the full batch)."""
    c = dict(DECODE_CONFIGS[name])
    if "seq_lens" in c:
        lens = list(c.pop("seq_lens"))
    else:
        lo, hi = c.pop("len_range")
        lens = draw_uniform_lengths(c["B"], lo, hi, seed)
        c["max_seq_len"] = hi
    if batch is not None:
        lens = lens[:batch]
        c["B"] = batch
    if poison is None:
        poison = name == "tiny_decode"
    return make_decode(seq_lens=lens, device=device, seed=seed, poison=poison,
                       name=name, **c)


# ---------------------------------------------------------------------------
# Prefill
# ---------------------------------------------------------------------------

@dataclass
class PrefillCache:
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor
    total_lens: list
    used_pages: list


def make_prefill_cache(total_lens, H_kv, D, P, *, device="cpu", seed=0,
                       pool_pages=None, poison=False):
    """A paged cache holding every sequence's full K/V (prefix + all chunks)."""
    gc = _cpu_gen(seed)
    total_lens = [int(x) for x in total_lens]
    max_pages = max(1, pages_for(max(total_lens + [1]), P))
    need = sum(pages_for(L, P) for L in total_lens)
    if pool_pages is None:
        pool_pages = max(need, 1)
    pt, used = build_page_table(total_lens, P, max_pages, pool_pages, gc)
    gd = _dev_gen(seed + 1, device)
    k_cache = torch.empty((pool_pages, P, H_kv, D), dtype=BF16, device=device)
    v_cache = torch.empty_like(k_cache)
    _fill_randn_bf16(k_cache, gd)
    _fill_randn_bf16(v_cache, gd)
    if poison:
        sl = torch.tensor(total_lens, dtype=torch.int32)
        poison_cache(k_cache, v_cache, pt, sl, used)
    return PrefillCache(k_cache, v_cache, pt.to(device), total_lens, used)


def make_prefill(cache: PrefillCache, q_lens, kv_lens, H_q, R, window, *,
                 device="cpu", seed=0, max_seq_len=None, name="",
                 rel_std=0.5, q_std=1.0):
    """One prefill call over ``cache``: sequence b has ``q_lens[b]`` new query
    tokens and ``kv_lens[b]`` keys in total (prefix + this chunk)."""
    q_lens = [int(x) for x in q_lens]
    kv_lens = [int(x) for x in kv_lens]
    T = sum(q_lens)
    D = cache.k_cache.shape[3]
    gd = _dev_gen(seed + 7, device)
    q = _randn((T, H_q, D), gd, device, BF16, std=q_std)
    rel = _randn((T, H_q, R), gd, device, torch.float32, std=rel_std)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    if max_seq_len is None:
        max_seq_len = max(kv_lens + [1])
    return PrefillInputs(q=q, cu_seqlens_q=cu.to(device), k_cache=cache.k_cache,
                         v_cache=cache.v_cache, page_table=cache.page_table,
                         seq_lens=torch.tensor(kv_lens, dtype=torch.int32).to(device),
                         rel_logits=rel, window=window, scale=1.0 / math.sqrt(D),
                         max_seq_len=max_seq_len, max_q_len=max(q_lens + [0]),
                         name=name)


CHUNKED_PREFILL = dict(n_seqs=4, seq_len=8192, chunk=2048, H_q=48, H_kv=16,
                       D=128, P=64, window=512, R=512)
# the same chunked prefill on a global layer: 8 KV heads, full causal, R = 1024
GLOBAL_PREFILL = dict(n_seqs=4, seq_len=8192, chunk=2048, H_q=48, H_kv=8,
                      D=128, P=64, window=0, R=1024)


def make_chunked_prefill(chunk_index, *, device="cpu", seed=0, cache=None, n_seqs=None,
                         cfg=None):
    """Call ``chunk_index`` (0..3) of a chunked-prefill workload (default the
    local-layer one): every sequence processes tokens [2048*c, 2048*(c+1))
    against the cached prefix.  ``n_seqs`` keeps only that many sequences (a
    smaller case of the same shape)."""
    c = CHUNKED_PREFILL if cfg is None else cfg
    n = c["n_seqs"] if n_seqs is None else int(n_seqs)
    if cache is None:
        cache = make_prefill_cache([c["seq_len"]] * n, c["H_kv"], c["D"],
                                   c["P"], device=device, seed=seed)
    q_lens = [c["chunk"]] * n
    kv_lens = [c["chunk"] * (chunk_index + 1)] * n
    return make_prefill(cache, q_lens, kv_lens, c["H_q"], c["R"], c["window"],
                        device=device, seed=seed + 100 * (chunk_index + 1),
                        max_seq_len=c["seq_len"],
                        name=f"chunked_prefill[{chunk_index}]"), cache


# ---------------------------------------------------------------------------
# 66-layer decode step
# ---------------------------------------------------------------------------

STACK = dict(n_layers=66, B=128, H_q=48, D=128, P=64, mean_len=2048, sigma=0.5,
             max_len=8192, local=dict(H_kv=16, window=512, R=512),
             glob=dict(H_kv=8, window=0, R=1024))


def is_global_layer(layer: int) -> bool:
    """Every 6th layer is global (11 of 66)."""
    return layer % 6 == 5


def draw_stack_lengths(seed=0):
    """Lognormal lengths with arithmetic mean 2048 (sigma 0.5), clipped to
    [1, 8192] and rounded."""
    s = STACK
    g = _cpu_gen(seed + 2000)
    mu = math.log(s["mean_len"]) - s["sigma"] ** 2 / 2
    z = torch.randn(s["B"], generator=g, dtype=torch.float64)
    L = torch.exp(mu + s["sigma"] * z).round().clamp(1, s["max_len"])
    return [int(x) for x in L.tolist()]
