"""GPU parity of paged (chunked) prefill, paged_prefill_attn, against the
oracle: the chunk's K/V written into the cache bit for bit, and the chunk's
queries attending through the block table, causal or not, within the bf16
tolerances.  Unfilled cache slots hold NaN, so any read past a sequence's
end, or any key a causal row must not see leaking in through P = 0 x NaN,
shows up."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(inp):
    return {k: getattr(inp, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "start_pos", "k_new", "v_new",
                                                 "q")}


def _check(inp, causal, out_dtype=torch.bfloat16, note=""):
    g = _dev(inp)
    ws = lib.Workspace(256)
    out = torch.empty(inp.q.shape, dtype=out_dtype, device=DEV)
    o, l = lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["start_pos"],
                                  k_new=g["k_new"], v_new=g["v_new"], causal=causal, scale=inp.scale, out=out,
                                  return_lse=True, workspace=ws)
    assert ws.status() == 0
    ek, ev = oracle.kv_append_chunk(inp.k_cache, inp.v_cache, inp.block_table, inp.start_pos, inp.k_new, inp.v_new)
    assert np.array_equal(g["k_cache"].cpu().view(torch.int16).numpy(), ek)
    assert np.array_equal(g["v_cache"].cpu().view(torch.int16).numpy(), ev)
    ro, rl = oracle.paged_prefill(inp.q, torch.from_numpy(ek).view(torch.bfloat16),
                                  torch.from_numpy(ev).view(torch.bfloat16), inp.block_table, inp.start_pos, causal,
                                  inp.scale)
    assert_out_close(o, ro, what="prefill out" + note)
    assert_lse_close(l, rl, what="prefill lse" + note)
    return o, l


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D,G,T", [(128, 4, 300), (128, 1, 37), (128, 2, 200), (64, 4, 256), (64, 2, 1), (64, 8, 150),
                                   (64, 1, 300), (128, 8, 129)])
def test_prefill_small(D, G, T, causal):
    """Starts 0 (a whole prompt), mid-block, on a tile edge, one past it, and
    long; chunks that end mid-block and mid-tile."""
    Hkv = 2
    cfg = workloads.PrefillConfig("s", 6, G * Hkv, Hkv, D, T, 16, 0, 0, 4, causal)
    inp = workloads.make_prefill_inputs(cfg, seed=21, start=[0, 5, 127, 128, 129, 1000])
    _check(inp, causal, note=f" D={D} G={G} T={T} causal={causal}")


@pytest.mark.parametrize("gain", [6.0, 40.0])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_peaked_scores(D, gain):
    """Queries scaled up so that a later key tile's scores exceed the running
    maximum by tens to hundreds of log2 units: the optimistic tiles' row-sum
    check fails and they are redone on the full path (causal, so the row
    limits apply too)."""
    cfg = workloads.PrefillConfig("p", 3, 8, 2, D, 260, 16, 0, 0, 2, True)
    inp = workloads.make_prefill_inputs(cfg, seed=24, start=[0, 129, 700])
    inp.q = (inp.q.float() * gain).to(torch.bfloat16)
    _check(inp, True, note=f" peaked D={D} gain={gain}")


def test_prefill_f32_output_and_preloaded_chunk():
    """out in f32, and k_new / v_new omitted: the chunk is already cached."""
    cfg = workloads.PrefillConfig("f", 3, 8, 2, 128, 200, 16, 0, 0, 2, True)
    inp = workloads.make_prefill_inputs(cfg, seed=22, start=[0, 33, 400])
    _check(inp, True, out_dtype=torch.float32, note=" f32")
    g = _dev(inp)
    lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["start_pos"],
                           k_new=g["k_new"], v_new=g["v_new"], causal=True, scale=inp.scale)
    o2, l2 = lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["start_pos"],
                                    causal=True, scale=inp.scale, return_lse=True)
    o1, l1 = lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["start_pos"],
                                    k_new=g["k_new"], v_new=g["v_new"], causal=True, scale=inp.scale,
                                    return_lse=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_chunked_prefill_equals_whole_prompt_on_gpu():
    """Prefilling a prompt in two chunks gives the rows of prefilling it in
    one pass (both on the GPU, each against the oracle too)."""
    S, T = 333, 400
    cfg = workloads.PrefillConfig("w", 2, 8, 2, 128, S + T, 16, 0, 0, 2, True)
    whole = workloads.make_prefill_inputs(cfg, seed=23, start=[0, 0])
    ow, lw = _check(whole, True, note=" whole")
    g = _dev(whole)
    # the same prompt again as chunk 1 (positions [0, S)) then chunk 2 ([S, S+T)),
    # into a fresh copy of the original cache
    kc = whole.k_cache.to(DEV)
    vc = whole.v_cache.to(DEV)
    zero = torch.zeros(2, dtype=torch.int32, device=DEV)
    lib.paged_prefill_attn(g["q"][:, :, :S].contiguous(), kc, vc, g["block_table"], zero,
                           k_new=g["k_new"][:, :, :S].contiguous(), v_new=g["v_new"][:, :, :S].contiguous(),
                           causal=True, scale=whole.scale)
    o2, l2 = lib.paged_prefill_attn(g["q"][:, :, S:].contiguous(), kc, vc, g["block_table"], zero + S,
                                    k_new=g["k_new"][:, :, S:].contiguous(), v_new=g["v_new"][:, :, S:].contiguous(),
                                    causal=True, scale=whole.scale, return_lse=True)
    assert (o2.float() - ow[:, :, S:].float()).abs().max().item() <= 2e-2
    assert (l2 - lw[:, :, S:]).abs().max().item() <= 1e-3


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_bad_start_and_bad_block(D):
    """A start position past the table and a block id outside the cache are
    reported, the sequence concerned is written as zeros, the others are
    exact (D 128 runs on CTA pairs, D 64 on the one-CTA kernel)."""
    cfg = workloads.PrefillConfig("b", 3, 8, 2, D, 50, 16, 0, 0, 2, True)
    inp = workloads.make_prefill_inputs(cfg, seed=24, start=[10, 20, 30])
    g = _dev(inp)
    sp = g["start_pos"].clone()
    sp[1] = -3  # reported: sequence 1 untouched, zeros out
    before = g["k_cache"].cpu().clone()
    ws = lib.Workspace(256)
    o, l = lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], sp, k_new=g["k_new"],
                                  v_new=g["v_new"], causal=True, scale=inp.scale, return_lse=True, workspace=ws)
    assert ws.status() == 5
    assert torch.all(o[1] == 0) and torch.all(torch.isneginf(l[1]))
    keep = [0, 2]
    ek, ev = oracle.kv_append_chunk(inp.k_cache, inp.v_cache, inp.block_table[keep], inp.start_pos[keep],
                                    inp.k_new[keep], inp.v_new[keep])
    got = g["k_cache"].cpu().view(torch.int16).numpy()
    assert np.array_equal(got, ek)  # sequence 1's blocks kept their old bits
    ro, rl = oracle.paged_prefill(inp.q[keep], torch.from_numpy(ek).view(torch.bfloat16),
                                  torch.from_numpy(ev).view(torch.bfloat16), inp.block_table[keep],
                                  inp.start_pos[keep], True, inp.scale)
    assert_out_close(o[keep], ro)
    assert_lse_close(l[keep], rl)
    # a table entry outside the cache: reported, no fault, no hang
    bt = g["block_table"].clone()
    bt[2, 1] = inp.num_blocks + 9
    ws.reset()
    lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], bt, g["start_pos"], causal=False, scale=inp.scale,
                           workspace=ws)
    assert ws.status() == 5
    del before


def test_prefill_full_workload_sampled_rows():
    """16 sequences each prefilling a 1024-token chunk after 0..7168 cached
    tokens, 32 query heads over 8 KV heads, D 128, causal (the configuration
    the benchmark times): the cache bit for bit, and windows of rows of every
    sequence against the oracle (a causal window of rows [i0, i0 + w) is the
    oracle's chunk of w rows starting at position start + i0)."""
    cfg = workloads.PREFILL_CONFIGS["prefill_chunk"]
    inp = workloads.make_prefill_inputs(cfg, seed=0)
    g = _dev(inp)
    ws = lib.Workspace(256)
    o, l = lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["start_pos"],
                                  k_new=g["k_new"], v_new=g["v_new"], causal=True, scale=inp.scale,
                                  return_lse=True, workspace=ws)
    assert ws.status() == 0
    ek, ev = oracle.kv_append_chunk(inp.k_cache, inp.v_cache, inp.block_table, inp.start_pos, inp.k_new, inp.v_new)
    assert np.array_equal(g["k_cache"].cpu().view(torch.int16).numpy(), ek)
    assert np.array_equal(g["v_cache"].cpu().view(torch.int16).numpy(), ev)
    kt, vt = torch.from_numpy(ek).view(torch.bfloat16), torch.from_numpy(ev).view(torch.bfloat16)
    w = 4
    for i0 in (0, 127, 128, 509, cfg.T - w):
        st = inp.start_pos + i0
        ro, rl = oracle.paged_prefill(inp.q[:, :, i0:i0 + w].contiguous(), kt, vt, inp.block_table, st, True,
                                      inp.scale)
        assert_out_close(o[:, :, i0:i0 + w], ro, what=f"prefill rows {i0}..")
        assert_lse_close(l[:, :, i0:i0 + w], rl, what=f"prefill lse rows {i0}..")
