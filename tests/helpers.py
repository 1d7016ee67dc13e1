"""Shared test helpers: run the CPU oracle on (a sample of) the same inputs the
GPU path sees, and compare within the stated tolerances.

Tolerances (bf16 outputs against the fp64 oracle): max-abs 2e-2 and mean-abs
2e-3; lse (fp32) within 2e-3 absolute.  Bit-exact checks compare raw bf16 bits.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle.ref import ref_decode, ref_prefill

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 2e-3


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def compact_pages(page_table, seq_lens, P, k_cache, v_cache):
    """Copy to the host only the pages the given sequences use, with a page
    table remapped onto the compact pool (same logical data)."""
    pt = page_table.cpu().numpy()
    sl = seq_lens.cpu().numpy()
    ids = []
    new_pt = np.zeros(pt.shape, dtype=np.int64)
    for r in range(pt.shape[0]):
        n = (int(sl[r]) + P - 1) // P
        for lp in range(n):
            new_pt[r, lp] = len(ids)
            ids.append(int(pt[r, lp]))
    if not ids:
        ids = [0]
    idx = torch.tensor(ids, dtype=torch.long, device=k_cache.device)
    kc = f64(k_cache.index_select(0, idx))
    vc = f64(v_cache.index_select(0, idx))
    return kc, vc, new_pt, sl.astype(np.int64)


def oracle_decode(inp, idx=None):
    """Oracle on sequences ``idx`` (default all) of a DecodeInputs."""
    if idx is None:
        idx = list(range(inp.B))
    sel = torch.tensor(idx, dtype=torch.long, device=inp.q.device)
    kc, vc, pt, sl = compact_pages(inp.page_table.index_select(0, sel),
                                   inp.seq_lens.index_select(0, sel), inp.page_size,
                                   inp.k_cache, inp.v_cache)
    return ref_decode(f64(inp.q.index_select(0, sel)), kc, vc, pt, sl,
                      f64(inp.rel_logits.index_select(0, sel)), inp.window, inp.scale)


def oracle_prefill(inp, seqs=None):
    """Oracle on sequences ``seqs`` (default all) of a PrefillInputs; returns
    (out, lse, token_index) with the packed token rows of those sequences."""
    cu = inp.cu_seqlens_q.cpu().numpy().astype(np.int64)
    B = inp.B
    if seqs is None:
        seqs = list(range(B))
    rows = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in seqs]) if seqs else np.zeros(0, int)
    new_cu = np.zeros(len(seqs) + 1, dtype=np.int64)
    for i, b in enumerate(seqs):
        new_cu[i + 1] = new_cu[i] + (cu[b + 1] - cu[b])
    sel = torch.tensor(seqs, dtype=torch.long, device=inp.q.device)
    kc, vc, pt, sl = compact_pages(inp.page_table.index_select(0, sel),
                                   inp.seq_lens.index_select(0, sel), inp.page_size,
                                   inp.k_cache, inp.v_cache)
    trow = torch.tensor(rows, dtype=torch.long, device=inp.q.device)
    out, lse = ref_prefill(f64(inp.q.index_select(0, trow)), new_cu, kc, vc, pt, sl,
                           f64(inp.rel_logits.index_select(0, trow)), inp.window, inp.scale)
    return out, lse, rows


def assert_close(gpu_out, ref_out, gpu_lse=None, ref_lse=None, max_abs=MAX_ABS,
                 mean_abs=MEAN_ABS, what=""):
    g = f64(gpu_out)
    assert g.shape == ref_out.shape, (g.shape, ref_out.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref_out)
    assert err.max() <= max_abs, f"{what}: max-abs {err.max():.3e} > {max_abs}"
    assert err.mean() <= mean_abs, f"{what}: mean-abs {err.mean():.3e} > {mean_abs}"
    if gpu_lse is not None and ref_lse is not None:
        gl = f64(gpu_lse)
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin), f"{what}: lse finiteness differs"
        if fin.any():
            le = np.abs(gl[fin] - ref_lse[fin])
            assert le.max() <= LSE_ABS, f"{what}: lse max-abs {le.max():.3e}"
        assert np.all(gl[~fin] == -np.inf)
    return float(err.max()), float(err.mean())


def bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy()
