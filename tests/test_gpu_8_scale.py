"""GPU parity for softmax scales of zero and below.

The definition of masked attention takes any finite scale (s = scale q.k +
mask, "MultiheadAttention fast path used 18 GB of VRAM", its SDPA section).
Two shortcuts in the kernels hold only for a positive scale: taking a tile's
row maximum over the raw scores and scaling it once, and certifying a tile by
the bound |q|_1 max|k| scale.  A scale of zero or below must route around
both.  These tests run the library through its C ABI with such scales and
compare it with the oracle at the same scale: attention on the tensor-core
instances (P over S at D = 64 and 128, P apart from S at the key-bound size)
and on the fp32 kernel, paged decode over bf16 and INT8 caches, and paged
prefill at D = 64 and 128."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _attn(inp, bounds):
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    mask = inp.mask.to(DEV) if inp.mask is not None else None
    B, Hkv, Pk, D = k.shape
    ws = lib.Workspace(lib.attn_fwd_workspace_size_for(B, Hkv, Pk, D) if bounds else 256)
    o, l = lib.attn_fwd(q, k, v, mask, inp.scale, workspace=ws)
    assert ws.status() == 0
    return o, l


@pytest.mark.parametrize("scale", [-0.125, 0.0])
@pytest.mark.parametrize("D", [64, 128])
def test_attn_scale_zero_and_negative(D, scale):
    """Several tiles, a padded tail, GQA and finite mask values: with scale 0
    the weights are the softmax of the mask alone."""
    inp = workloads.make_attn(2, 4, 2, 200, 333, D, dtype=torch.bfloat16, n_pad=[0, 45], seed=81)
    inp.mask[0, 100:110] = 1.5
    inp.mask[1, 7] = -3.0
    inp.scale = scale
    o, l = _attn(inp, bounds=True)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, scale)
    assert_out_close(o, ro, what=f"D={D} scale={scale}")
    assert_lse_close(l, rl, what=f"lse D={D} scale={scale}")


def test_attn_negative_scale_at_the_key_bound_size():
    """D = 64 at B Hq Pq Pk D = 2^36, where attn_fwd computes per-tile key
    bounds and runs the instance with P apart from S: sampled rows of every
    head."""
    inp = workloads.make_attn(1, 16, 8, 8192, 8192, 64, dtype=torch.bfloat16, n_pad=300, seed=82)
    inp.scale = -0.125
    o, l = _attn(inp, bounds=True)
    rows = sample_rows(1, 16, 8192, 256, seed=13)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale, rows=rows)
    idx = torch.from_numpy(rows).to(DEV)
    assert_out_close(o.reshape(-1, 64)[idx], ro, what="key-bound size, scale -1/8")
    assert_lse_close(l.reshape(-1)[idx], rl)


def test_attn_f32_negative_scale():
    inp = workloads.make_attn(1, 2, 2, 150, 260, 64, dtype=torch.float32, n_pad=20, seed=83)
    inp.scale = -0.3
    o, l = _attn(inp, bounds=False)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro, fp32_inputs=True, what="f32 scale -0.3")
    assert_lse_close(l, rl)


@pytest.mark.parametrize("scale", [-0.1, 0.0])
@pytest.mark.parametrize("D", [128, 64])
def test_paged_decode_scale_zero_and_negative(D, scale):
    cfg = workloads.DecodeConfig("n", 5, 8, 2, D, 16, 0, 1500, 4)
    d = workloads.make_decode_inputs(cfg, seed=84, ctx=[0, 16, 600, 1024, 1500])
    d.scale = scale
    g = {k: getattr(d, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "pos", "ctx_lens", "k_new", "v_new",
                                            "q")}
    ws = lib.Workspace(lib.paged_decode_workspace_size(cfg.B, cfg.Hq, d.block_table.shape[1], 16, D))
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"], workspace=ws)
    out, lse = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], scale,
                                     return_lse=True, workspace=ws)
    assert ws.status() == 0
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    ro, rl = oracle.paged_decode(d.q, torch.from_numpy(ek).view(torch.bfloat16),
                                 torch.from_numpy(ev).view(torch.bfloat16), d.block_table, d.ctx_lens, scale)
    assert_out_close(out, ro, what=f"decode D={D} scale={scale}")
    assert_lse_close(lse, rl, what=f"decode lse D={D} scale={scale}")


@pytest.mark.parametrize("scale", [-0.1, 0.0])
def test_q8_decode_scale_zero_and_negative(scale):
    cfg = workloads.DecodeConfig("n8", 5, 8, 2, 128, 16, 0, 1500, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=85, ctx=[0, 16, 600, 1024, 1500])
    g = {k: getattr(d, k).to(DEV) for k in ("kq_cache", "vq_cache", "k_scale", "v_scale", "block_table", "pos",
                                            "ctx_lens", "k_new", "v_new", "q")}
    ws = lib.Workspace(lib.paged_decode_workspace_size(cfg.B, cfg.Hq, d.block_table.shape[1], 16, cfg.D))
    lib.kv_append_q8(g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"], g["block_table"], g["pos"],
                     g["k_new"], g["v_new"], workspace=ws)
    out, lse = lib.paged_decode_attn_q8(g["q"], g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"],
                                        g["block_table"], g["ctx_lens"], scale, return_lse=True, workspace=ws)
    assert ws.status() == 0
    kq, vq, ks, vs = oracle.kv_append_q8(d.kq_cache, d.vq_cache, d.k_scale, d.v_scale, d.block_table, d.pos,
                                         d.k_new, d.v_new)
    ro, rl = oracle.paged_decode_q8(d.q, kq, vq, ks, vs, d.block_table, d.ctx_lens, scale)
    assert_out_close(out, ro, what=f"q8 decode scale={scale}")
    assert_lse_close(lse, rl, what=f"q8 decode lse scale={scale}")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_paged_prefill_negative_scale(D, causal):
    cfg = workloads.PrefillConfig("n", 3, 8, 2, D, 200, 16, 0, 0, 2, causal)
    inp = workloads.make_prefill_inputs(cfg, seed=86, start=[0, 37, 300])
    scale = -0.1
    g = {k: getattr(inp, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "start_pos", "k_new", "v_new",
                                              "q")}
    ws = lib.Workspace(256)
    o, l = lib.paged_prefill_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["start_pos"],
                                  k_new=g["k_new"], v_new=g["v_new"], causal=causal, scale=scale, return_lse=True,
                                  workspace=ws)
    assert ws.status() == 0
    ek, ev = oracle.kv_append_chunk(inp.k_cache, inp.v_cache, inp.block_table, inp.start_pos, inp.k_new, inp.v_new)
    ro, rl = oracle.paged_prefill(inp.q, torch.from_numpy(ek).view(torch.bfloat16),
                                  torch.from_numpy(ev).view(torch.bfloat16), inp.block_table, inp.start_pos, causal,
                                  scale)
    assert_out_close(o, ro, what=f"prefill D={D} causal={causal}")
    assert_lse_close(l, rl, what=f"prefill lse D={D} causal={causal}")
    assert np.all(np.isfinite(o.float().cpu().numpy()))
