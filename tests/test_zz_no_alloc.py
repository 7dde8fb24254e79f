"""paged_decode_attn_noalloc: the paged decode for callers that cannot
allocate device memory (a plugin handed only its input and output buffers, or
a loop whose device footprint must stay fixed).  Its split-K scratch is a
20 MiB array built into the library.

Through the C ABI, two calls in a row (different batches, so the second runs
over what the first left in the shared scratch) must match the workspace
entry point paged_decode_attn within the bf16 tolerances, and the oracle's
decode directly on a few sequences of each batch; the calls must not grow
device memory.  This file is collected last; it passes alone in a fresh
process and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close
from masked_attention_paged_gb300 import AttnKVCache, AttnTensor

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _desc(t):
    d = AttnTensor()
    d.data, d.dtype, d.ndim = t.data_ptr(), 1 if t.dtype == torch.bfloat16 else 0, t.dim()
    for i in range(t.dim()):
        d.shape[i], d.stride[i] = t.shape[i], t.stride(i)
    return d


def _cache(k, v):
    c = AttnKVCache()
    c.k, c.v, c.dtype = k.data_ptr(), v.data_ptr(), 1
    c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim = k.shape[0], k.shape[1], k.shape[2], k.shape[3]
    return c


def _noalloc(L, q, kc, vc, bt, lens, scale, out, lse, status):
    return L.paged_decode_attn_noalloc(ctypes.byref(_desc(q)), ctypes.byref(_cache(kc, vc)), bt.data_ptr(),
                                       bt.stride(0), bt.shape[1], lens.data_ptr(), scale, ctypes.byref(_desc(out)),
                                       lse.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _case(cfg, seed):
    d = workloads.make_decode_inputs(cfg, seed=seed)
    g = {k: getattr(d, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "pos", "ctx_lens", "k_new",
                                            "v_new", "q")}
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"])
    ref_o, ref_l = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"],
                                         d.scale, return_lse=True)
    return d, g, ref_o, ref_l


def _oracle_rows(d, seqs):
    """The oracle's decode of sequences `seqs`, over the cache after the
    oracle's own append of each sequence's new token (CPU inputs only)."""
    kc, vc = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    kc, vc = torch.from_numpy(kc).view(torch.bfloat16), torch.from_numpy(vc).view(torch.bfloat16)
    return oracle.paged_decode(d.q[seqs], kc, vc, d.block_table[seqs], d.ctx_lens[seqs], d.scale)


def test_noalloc_matches_workspace_entry_point_twice():
    L = lib.load()
    cases = [_case(workloads.DECODE_CONFIGS["decode"], 0),
             _case(workloads.DecodeConfig("second", 9, 32, 8, 128, 16, 0, 3000, 7), 5)]
    status = torch.ones(1, dtype=torch.int32, device=DEV)
    for n, (d, g, ref_o, ref_l) in enumerate(cases):
        out = torch.empty_like(ref_o)
        lse = torch.empty_like(ref_l)
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        reserved0 = torch.cuda.memory_reserved()
        free0 = torch.cuda.mem_get_info()[0]
        st = _noalloc(L, g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], d.scale, out, lse,
                      status)
        torch.cuda.synchronize()
        assert st == 0, L.attn_status_string(st)
        assert int(status.item()) == 0
        # nothing through torch's allocator ...
        assert torch.cuda.memory_allocated() == alloc0 and torch.cuda.memory_reserved() == reserved0
        # ... nor past it.  CUDA loads the library's device code onto a GPU lazily, at
        # its first use there, and the scratch array comes with that code: the first
        # call in a process may see that one-time load (20 MiB), later calls nothing
        # (a small allowance for whatever else the driver does meanwhile).
        drop = free0 - torch.cuda.mem_get_info()[0]
        assert drop <= (2 << 20) + (0 if n else (20 << 20)), drop
        diff = (out.float() - ref_o.float()).abs()
        assert diff.max().item() <= 2e-2 and diff.mean().item() <= 2e-3
        assert (lse - ref_l).abs().max().item() <= 1e-3
        # and directly against the oracle on a few sequences (the longest among them)
        seqs = sorted({0, d.cfg.B - 1, int(torch.argmax(d.ctx_lens)), d.cfg.B // 2})
        ro, rl = _oracle_rows(d, seqs)
        idx = torch.tensor(seqs, device=DEV)
        assert_out_close(out[idx], ro, what=f"noalloc {d.cfg.name}")
        assert_lse_close(lse[idx], rl, what=f"noalloc lse {d.cfg.name}")


def test_noalloc_rejects_a_call_larger_than_its_scratch():
    L = lib.load()
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(8, 8, 16, 128, dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros(64, 2000, dtype=torch.int32, device=DEV)  # contexts up to 32000 tokens: 68 MB of partials
    lens = torch.ones(64, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    lse = torch.empty(64, 32, dtype=torch.float32, device=DEV)
    st = _noalloc(L, q, kc, kc, bt, lens, 0.1, out, lse, torch.zeros(1, dtype=torch.int32, device=DEV))
    assert st == 6  # ATTN_ERR_WORKSPACE


def test_noalloc_reports_bad_block_ids_in_its_status():
    L = lib.load()
    cfg = workloads.DecodeConfig("bad", 3, 8, 2, 128, 16, 50, 200, 2)
    d = workloads.make_decode_inputs(cfg, seed=3)
    g = {k: getattr(d, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "ctx", "q")}
    bt = g["block_table"].clone()
    bt[1, 0] = -3
    out = torch.empty_like(g["q"])
    lse = torch.empty(3, 8, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert _noalloc(L, g["q"], g["k_cache"], g["v_cache"], bt, g["ctx"], d.scale, out, lse, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 1 << 5
    # the next good call starts from a clean status word
    assert _noalloc(L, g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx"], d.scale, out, lse,
                    status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
