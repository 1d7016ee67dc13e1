"""Host logic of the benchmark's end-to-end harness on CPU: a step's inputs
(q, rel_logits, page_table, seq_lens) and outputs (out, lse) travel packed in
one flat buffer each; the views into it must be aligned, disjoint and carry
the tensors unchanged."""

from __future__ import annotations

import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _specs(B=5, H_q=12, H_kv=4, D=64, R=33, pages=7):
    return [(torch.bfloat16, (B, H_q, D)), (torch.float32, (B, H_q, R)),
            (torch.int32, (B, pages)), (torch.int32, (B,))]


def test_packed_views_are_aligned_and_disjoint():
    specs = _specs()
    nbytes = bench._packed_bytes(specs)
    buf = torch.zeros(nbytes, dtype=torch.uint8)
    views, used = bench._packed_views(buf, specs)
    assert used == nbytes
    base = buf.data_ptr()
    spans = []
    for v, (dtype, shape) in zip(views, specs):
        assert v.dtype == dtype and tuple(v.shape) == tuple(shape) and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0  # q and rel_logits are read by 16-byte bulk copies
        spans.append((off, off + v.numel() * v.element_size()))
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0  # in order, no overlap
    assert spans[-1][1] <= nbytes


def test_packed_round_trip_is_bit_exact():
    specs = _specs()
    g = torch.Generator().manual_seed(3)
    src = [torch.randn(specs[0][1], generator=g).to(torch.bfloat16),
           torch.randn(specs[1][1], generator=g),
           torch.randint(-1, 1000, specs[2][1], generator=g, dtype=torch.int32),
           torch.randint(0, 5000, specs[3][1], generator=g, dtype=torch.int32)]
    buf = torch.empty(bench._packed_bytes(specs), dtype=torch.uint8)
    views, _ = bench._packed_views(buf, specs)
    for v, t in zip(views, src):
        v.copy_(t)
    # one flat copy moves everything (the harness's single host-to-device copy)
    moved = buf.clone()
    back, _ = bench._packed_views(moved, specs)
    for v, t in zip(back, src):
        assert torch.equal(v.view(torch.uint8) if v.dtype == torch.bfloat16 else v,
                           t.view(torch.uint8) if t.dtype == torch.bfloat16 else t)


def test_packed_sizes_of_the_local_decode_step():
    """64 sequences, 48/16 heads, D = 128, R = 512, page-table rows of 128:
    every piece is already a multiple of 256 bytes, so the upload is exactly
    the tensors' bytes."""
    specs = [(torch.bfloat16, (64, 48, 128)), (torch.float32, (64, 48, 512)),
             (torch.int32, (64, 128)), (torch.int32, (64,))]
    exact = 64 * 48 * 128 * 2 + 64 * 48 * 512 * 4 + 64 * 128 * 4 + 64 * 4
    assert bench._packed_bytes(specs) == exact == 7110912


def test_source_hash_ignores_comments_and_layout(tmp_path, monkeypatch):
    code = 'int f(int x) {\n  return x + 1;  // one\n}\nconst char* s = "// kept /* too */";\n'
    edited = '/* header */\nint f(int x) {\n    return x + 1;\n}\n// note\nconst char* s = "// kept /* too */";\n'
    changed = code.replace("x + 1", "x + 2")
    for name, text in (("a.cu", code), ("b.cu", edited), ("c.cu", changed)):
        (tmp_path / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.source_hash(["a.cu"]) == bench.source_hash(["b.cu"])
    assert bench.source_hash(["a.cu"]) != bench.source_hash(["c.cu"])
    assert '"// kept /* too */"' in bench.strip_c_comments(code)


def test_traffic_records_match_the_current_sources():
    """Every committed DRAM-traffic record was taken on the kernel code as it
    stands (a stale record would make the bench report traffic null)."""
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    for key, rec in recs.items():
        kernel = key.split(":")[0]
        assert rec["source_hash"] == bench.source_hash(bench.KERNEL_SOURCES[kernel]), key
