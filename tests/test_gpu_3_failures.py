"""Failure detection on the GPU without faulting it.

A kernel waits on a barrier phase nothing completes: the library's wait
guard must give up after the requested limit, record ATTN_ERR_TIMEOUT in the
workspace status word, and leave the CUDA context usable (a normal call right
after returns correct results).  Out-of-range block ids and positions are
covered in test_gpu_1_paged.py."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_out_close

pytestmark = pytest.mark.gpu


def test_wait_guard_times_out_and_context_survives():
    L = lib.load()
    ws = lib.Workspace(256)
    stream = torch.cuda.current_stream().cuda_stream
    st = L.attn_selftest_wait_timeout(ws.ptr, ws.nbytes, 20000, stream)  # 20 ms
    assert st == 0
    assert ws.status() == 4  # ATTN_ERR_TIMEOUT
    ws.reset()
    assert ws.status() == 0
    # the context is intact: a real call runs and is right
    inp = workloads.make_attn(1, 2, 2, 130, 200, 64, dtype=torch.bfloat16, n_pad=9, seed=21)
    o, l = lib.attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.mask.cuda(), inp.scale, workspace=ws)
    assert ws.status() == 0
    ro, _ = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro)


def test_selftest_rejects_bad_limits():
    L = lib.load()
    ws = lib.Workspace(256)
    stream = torch.cuda.current_stream().cuda_stream
    assert L.attn_selftest_wait_timeout(ws.ptr, ws.nbytes, 0, stream) == 1
    assert L.attn_selftest_wait_timeout(ws.ptr, ws.nbytes, 2000000, stream) == 1
    assert L.attn_selftest_wait_timeout(None, 256, 1000, stream) == 6
