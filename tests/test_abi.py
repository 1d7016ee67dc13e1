"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its host-only helpers (split plan, workspace size, error
strings, argument validation) behave as documented."""

from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "inkling_rel_attn.h")


@pytest.fixture(scope="module")
def lib():
    from paged_attention_relative_attn_gb300 import build, _lib
    build.build()
    return _lib


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(inkling_rel_attn_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    from paged_attention_relative_attn_gb300 import _lib
    assert declared_functions() == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(so, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    for name in declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert len(lib.inkling_rel_attn_error_string(code)) > 5
    assert "unknown" in lib.inkling_rel_attn_error_string(-99)
    assert lib.inkling_rel_attn_version() >= 100


def test_split_plan_local_and_global(lib):
    # local-layer decode: 64 x 16 pairs over 512 keys already fill the GPU
    assert lib.inkling_rel_attn_choose_splits(64, 16, 512, 8192, 152) == 1
    # global-layer decode: 32 x 8 pairs over up to 32768 keys -> 1024-key splits
    assert lib.inkling_rel_attn_choose_splits(32, 8, 0, 32768, 152) == 32
    # few pairs over a window: split the window, never below 256 keys
    assert lib.inkling_rel_attn_choose_splits(1, 16, 512, 8192, 152) == 2
    # tiny: one split
    assert lib.inkling_rel_attn_choose_splits(2, 2, 32, 100, 152) == 1
    # never above 128 splits
    assert lib.inkling_rel_attn_choose_splits(1, 1, 0, 1 << 20, 152) == 128
    # num_sms <= 0 means 152
    assert (lib.inkling_rel_attn_choose_splits(32, 8, 0, 32768, 0)
            == lib.inkling_rel_attn_choose_splits(32, 8, 0, 32768, 152))


def test_workspace_size(lib):
    assert lib.inkling_rel_attn_decode_workspace_size(64, 48, 16, 128, 512, 8192, 0, 152) == 0
    S = lib.inkling_rel_attn_choose_splits(32, 8, 0, 32768, 152)
    rows = 32 * 48 * S
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert (lib.inkling_rel_attn_decode_workspace_size(32, 48, 8, 128, 0, 32768, 0, 152)
            == 256 + r256(rows * 128 * 4) + r256(rows * 4))
    # forced splits are clamped to one per 64 keys
    assert lib.inkling_rel_attn_decode_workspace_size(1, 4, 2, 64, 0, 100, 50, 152) == \
        256 + r256(1 * 4 * 2 * 64 * 4) + r256(1 * 4 * 2 * 4)
    assert lib.inkling_rel_attn_prefill_workspace_size(8192, 48, 128) == 0


def _decode_rc(lib, **over):
    a = dict(q=16, k_cache=16, v_cache=16, page_table=4, page_table_stride=4, seq_lens=4,
             rel_logits=4, B=2, H_q=4, H_kv=2, D=64, page_size=16, num_pages=16, R=32, window=32,
             scale=0.125, max_seq_len=100, out=16, lse_out=None, workspace=None,
             workspace_bytes=0, num_splits=0, device_error=None, stream=None)
    a.update(over)
    return lib.inkling_rel_attn_decode(**a)


def test_decode_argument_validation(lib):
    # shape errors are reported before any device is touched
    assert _decode_rc(lib, D=96) == -1
    assert _decode_rc(lib, H_q=5) == -1
    assert _decode_rc(lib, H_q=34, H_kv=2) == -1      # group of 17 > 16
    assert _decode_rc(lib, page_size=24) == -1
    assert _decode_rc(lib, R=0) == -1
    assert _decode_rc(lib, B=-1) == -1
    assert _decode_rc(lib, q=None) == -1
    assert _decode_rc(lib, B=0) == 0                  # empty batch: nothing to do
    assert _decode_rc(lib, q=24) == -2                # 8-byte aligned only
    assert _decode_rc(lib, seq_lens=6) == -2


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-device answer")
def test_decode_without_device_reports_device_error(lib):
    assert _decode_rc(lib) == -4


def test_prefill_argument_validation(lib):
    a = dict(q=16, cu_seqlens_q=4, k_cache=16, v_cache=16, page_table=4, page_table_stride=4,
             seq_lens=4, rel_logits=16, B=1, T=4, max_q_len=4, H_q=4, H_kv=2, D=64,
             page_size=16, num_pages=4, R=32, window=0, scale=0.1, max_seq_len=64, out=16,
             lse_out=None, workspace=None, workspace_bytes=0, device_error=None, stream=None)
    assert lib.inkling_rel_attn_prefill(**{**a, "R": 30}) == -1
    assert lib.inkling_rel_attn_prefill(**{**a, "rel_logits": 8}) == -2
    assert lib.inkling_rel_attn_prefill(**{**a, "T": 0}) == 0


def test_kv_append_argument_validation(lib):
    a = dict(k_new=16, v_new=16, cu_seqlens_q=4, seq_lens=4, page_table=4, page_table_stride=4,
             B=2, T=2, H_kv=2, D=64, page_size=16, num_pages=8, k_cache=16, v_cache=16,
             device_error=None, stream=None)
    rc = lambda **o: lib.inkling_rel_attn_kv_append(**{**a, **o})  # noqa: E731
    assert rc(D=96) == -1
    assert rc(page_size=24) == -1
    assert rc(num_pages=0) == -1
    assert rc(H_kv=0) == -1
    assert rc(B=-1) == -1
    assert rc(T=0) == 0                 # nothing to write
    assert rc(B=0) == 0
    assert rc(k_new=None) == -1
    assert rc(k_cache=24) == -2         # 16-byte alignment
    assert rc(seq_lens=6) == -2


def test_kv_conv_append_argument_validation(lib):
    a = dict(k_new=16, v_new=16, cu_seqlens_q=4, seq_lens=4, page_table=4, page_table_stride=4,
             conv_w_k=4, conv_w_v=4, width=4, conv_state_k=16, conv_state_v=16, state_slots=4,
             num_slots=3, B=2, T=2, max_q_len=2, H_kv=2, D=64, page_size=16, num_pages=8,
             k_cache=16, v_cache=16, device_error=None, stream=None)
    rc = lambda **o: lib.inkling_rel_attn_kv_conv_append(**{**a, **o})  # noqa: E731
    assert rc(width=0) == -1
    assert rc(width=9) == -1
    assert rc(D=96) == -1
    assert rc(page_size=24) == -1
    assert rc(num_slots=0) == -1        # a state pool is needed when width > 1
    assert rc(max_q_len=-1) == -1
    assert rc(B=0) == 0 and rc(T=0) == 0 and rc(max_q_len=0) == 0
    assert rc(conv_w_k=None) == -1
    assert rc(conv_state_v=None) == -1
    assert rc(conv_state_k=24) == -2    # 16-byte alignment
    assert rc(conv_w_v=2) == -2
    # width 1 needs no state: with the state pointers NULL the call gets as far
    # as the alignment check (it would stop at -1 if they were required)
    assert rc(width=1, num_slots=0, conv_state_k=None, conv_state_v=None, state_slots=None,
              k_cache=24) == -2


def test_decode_multi_validation_and_workspace(lib):
    a = dict(q=16, k_cache=16, v_cache=16, page_table=4, page_table_stride=4, seq_lens=4,
             rel_logits=4, B=2, q_len=4, H_q=4, H_kv=2, D=64, page_size=16, num_pages=16, R=32,
             window=32, scale=0.125, max_seq_len=100, out=16, lse_out=None, workspace=None,
             workspace_bytes=0, num_splits=0, device_error=None, stream=None)
    rc = lambda **o: lib.inkling_rel_attn_decode_multi(**{**a, **o})  # noqa: E731
    assert rc(q_len=0) == -1
    assert rc(q_len=65) == -1
    assert rc(max_seq_len=3) == -1          # fewer keys than new tokens
    assert rc(D=96) == -1
    assert rc(B=0) == 0
    assert rc(q=24) == -2
    # q_len = 1 is plain decode: same workspace
    for args in ((32, 48, 8, 128, 0, 32768, 0, 152), (64, 48, 16, 128, 512, 8192, 0, 152),
                 (1, 4, 2, 64, 0, 100, 50, 152)):
        B, H_q, H_kv, D, W_, L, S, sms = args
        assert (lib.inkling_rel_attn_decode_multi_workspace_size(B, 1, H_q, H_kv, D, W_, L, S, sms)
                == lib.inkling_rel_attn_decode_workspace_size(B, H_q, H_kv, D, W_, L, S, sms))
    # several tokens: partials for every (token, head, split)
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    ws = lib.inkling_rel_attn_decode_multi_workspace_size(2, 4, 12, 2, 128, 0, 40000, 8, 152)
    assert ws == 256 + r256(2 * 4 * 12 * 8 * 128 * 4) + r256(2 * 4 * 12 * 8 * 4)
