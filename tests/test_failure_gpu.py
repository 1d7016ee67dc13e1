"""Failure handling on the GPU without a fault: a bounded wait that is made
to run out reports INKLING_DEVERR_TIMEOUT and the context stays usable."""

from __future__ import annotations

import time

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_attention_relative_attn_gb300 import build, _lib
    build.build()
    return _lib


def test_wait_timeout_is_reported_and_context_survives(lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    rc = lib.inkling_rel_attn_selftest_timeout(err.data_ptr(), 50,
                                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert rc == 0
    assert int(err.item()) == 4          # INKLING_DEVERR_TIMEOUT
    assert dt < 5.0                      # it gave up on its own
    # the context is intact: a normal decode still runs and is finite
    import paged_attention_relative_attn_gb300 as ira
    inp = W.make_decode_config("tiny_decode", device="cuda")
    out, _ = ira.decode_inputs(inp)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


def test_selftest_argument_checks(lib):
    assert lib.inkling_rel_attn_selftest_timeout(None, 50, None) == -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.inkling_rel_attn_selftest_timeout(err.data_ptr(), 0, None) == -1
