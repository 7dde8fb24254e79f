"""GPU parity of the INT8 KV cache calls (memory accounting page, section 18):
kv_append_q8's codes and scales bit for bit against the oracle's quantiser,
and paged_decode_attn_q8 against the oracle's decode over the dequantised
cache within the bf16 tolerances, at small ragged sizes and at the full
decode workload.  Unfilled slots hold a NaN scale, so reading one shows."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(d):
    return {k: getattr(d, k).to(DEV) for k in ("kq_cache", "vq_cache", "k_scale", "v_scale", "block_table", "pos",
                                               "ctx_lens", "ctx", "k_new", "v_new", "q")}


def _append_decode_check(d, note=""):
    g = _dev(d)
    ws = lib.Workspace(lib.paged_decode_workspace_size(d.cfg.B, d.cfg.Hq, d.block_table.shape[1], 16, d.cfg.D))
    lib.kv_append_q8(g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"], g["block_table"], g["pos"],
                     g["k_new"], g["v_new"], workspace=ws)
    out, lse = lib.paged_decode_attn_q8(g["q"], g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"],
                                        g["block_table"], g["ctx_lens"], d.scale, return_lse=True, workspace=ws)
    assert ws.status() == 0
    kq, vq, ks, vs = oracle.kv_append_q8(d.kq_cache, d.vq_cache, d.k_scale, d.v_scale, d.block_table, d.pos,
                                         d.k_new, d.v_new)
    np.testing.assert_array_equal(g["kq_cache"].cpu().numpy(), kq)
    np.testing.assert_array_equal(g["vq_cache"].cpu().numpy(), vq)
    # scales as bits (NaN sentinels included)
    np.testing.assert_array_equal(g["k_scale"].cpu().numpy().view(np.int32), ks.view(np.int32))
    np.testing.assert_array_equal(g["v_scale"].cpu().numpy().view(np.int32), vs.view(np.int32))
    ro, rl = oracle.paged_decode_q8(d.q, kq, vq, ks, vs, d.block_table, d.ctx_lens, d.scale)
    assert_out_close(out, ro, what="q8 decode out" + note)
    assert_lse_close(lse, rl, what="q8 decode lse" + note)


@pytest.mark.parametrize("D,G", [(128, 4), (128, 1), (128, 2), (128, 8), (64, 4), (64, 2), (64, 1), (64, 8)])
def test_q8_append_and_decode_small(D, G):
    Hkv = 2
    cfg = workloads.DecodeConfig("q", 9, G * Hkv, Hkv, D, 16, 0, 1500, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=51, ctx=[0, 15, 16, 511, 512, 1023, 1024, 1300, 1500])
    _append_decode_check(d, f" D={D} G={G}")


def test_q8_long_context():
    """40 and 33 splits of 1024 tokens: the split merge's second pass."""
    cfg = workloads.DecodeConfig("l", 3, 8, 2, 128, 16, 0, 40000, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=57, ctx=[40000, 33000, 100])
    _append_decode_check(d, " long")


def test_q8_full_decode_workload():
    d = workloads.make_decode_inputs_q8(workloads.DECODE_CONFIGS["decode"], seed=0)
    _append_decode_check(d, " full")


def test_q8_append_zero_rows_idle_and_bad_positions():
    cfg = workloads.DecodeConfig("q", 4, 8, 2, 128, 16, 0, 100, 2)
    d = workloads.make_decode_inputs_q8(cfg, seed=52, ctx=[3, 30, 60, 90])
    d.k_new[0] = 0  # all-zero rows: scale 0, codes 0
    g = _dev(d)
    pos = g["pos"].clone()
    pos[1] = -1  # idle
    pos[2] = 16 * d.block_table.shape[1]  # past the table
    ws = lib.Workspace(256)
    lib.kv_append_q8(g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"], g["block_table"], pos,
                     g["k_new"], g["v_new"], workspace=ws)
    assert ws.status() == 5
    p2 = d.pos.clone()
    p2[1] = -1
    p2[2] = -1
    kq, vq, ks, vs = oracle.kv_append_q8(d.kq_cache, d.vq_cache, d.k_scale, d.v_scale, d.block_table, p2,
                                         d.k_new, d.v_new)
    np.testing.assert_array_equal(g["kq_cache"].cpu().numpy(), kq)
    np.testing.assert_array_equal(g["k_scale"].cpu().numpy().view(np.int32), ks.view(np.int32))
    blk, slot = int(d.block_table[0, int(d.pos[0]) // 16]), int(d.pos[0]) % 16
    assert np.all(ks[blk, :, slot] == 0) and not kq[blk, :, slot].any()


def test_q8_decode_tracks_the_bf16_decode():
    """Quantising a bf16 cache with the library and decoding it stays close to
    decoding the bf16 cache: the INT8 codes keep about 7 bits per element."""
    cfg = workloads.DecodeConfig("r", 8, 32, 8, 128, 16, 200, 500, 4)
    d = workloads.make_decode_inputs(cfg, seed=53)
    g = {k: getattr(d, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "pos", "ctx_lens", "k_new",
                                           "v_new", "q")}
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"])
    ref = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], d.scale)
    # the whole bf16 cache quantised row by row through kv_append_q8, one slot at a time per sequence
    nb, H, bs, D = d.k_cache.shape
    kq = torch.zeros(nb, H, bs, D, dtype=torch.int8, device=DEV)
    vq = torch.zeros_like(kq)
    ks = torch.full((nb, H, bs), float("nan"), device=DEV)
    vs = torch.full_like(ks, float("nan"))
    for t in range(int(d.ctx_lens.max())):
        pos = torch.where(d.ctx_lens > t, torch.full_like(d.ctx_lens, t), torch.full_like(d.ctx_lens, -1))
        bt = d.block_table.clone()
        kn = torch.zeros(cfg.B, H, D, dtype=torch.bfloat16)
        vn = torch.zeros_like(kn)
        for b in range(cfg.B):
            if t < int(d.ctx_lens[b]):
                blk = int(bt[b, t // 16])
                kn[b] = g["k_cache"][blk, :, t % 16].cpu()
                vn[b] = g["v_cache"][blk, :, t % 16].cpu()
        lib.kv_append_q8(kq, vq, ks, vs, g["block_table"], pos.to(DEV).to(torch.int32), kn.to(DEV), vn.to(DEV))
    out = lib.paged_decode_attn_q8(g["q"], kq, vq, ks, vs, g["block_table"], g["ctx_lens"], d.scale)
    err = (out.float() - ref.float()).abs()
    assert err.max().item() < 3e-2 and err.mean().item() < 3e-3


def _decode_only_check(d, scale, note, abs_floor=0.0):
    """Decode the cache as given (no append) with float32 output, against the
    oracle within a bound taken from the arithmetic: a softmax weight rounded
    to fp16 is off by at most 2^-11 of itself, so an output element is off by
    at most 2^-11 sum_t p_t |v_t| / l, which the oracle gives when it decodes
    |V|; twice that, plus a floor of 1e-6 of the largest such sum."""
    g = _dev(d)
    out = torch.empty(d.q.shape, dtype=torch.float32, device=DEV)
    ws = lib.Workspace(lib.paged_decode_workspace_size(d.cfg.B, d.cfg.Hq, d.block_table.shape[1], 16, d.cfg.D))
    _, lse = lib.paged_decode_attn_q8(g["q"], g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"],
                                      g["block_table"], g["ctx"], scale, out=out, return_lse=True, workspace=ws)
    assert ws.status() == 0
    kq, vq, ks, vs = d.kq_cache.numpy(), d.vq_cache.numpy(), d.k_scale.numpy(), d.v_scale.numpy()
    ro, rl = oracle.paged_decode_q8(d.q, kq, vq, ks, vs, d.block_table, d.ctx, scale)
    ra, _ = oracle.paged_decode_q8(d.q, kq, np.abs(vq), ks, vs, d.block_table, d.ctx, scale)
    err = np.abs(out.cpu().numpy().astype(np.float64) - ro)
    bound = 2.0 ** -10 * ra + 1e-6 * ra.max() + abs_floor
    assert np.all(err <= bound), f"{note}: worst err/bound {(err / bound).max():.3g}"
    assert_lse_close(lse, rl, what="q8 decode lse " + note)


@pytest.mark.parametrize("gain", [8.0, 40.0])
def test_q8_decode_peaked_scores(gain):
    """Queries scaled up (scores over tens to hundreds of log2 units): the
    running maximum and the value-weight reference move within and across
    blocks, and the weights are nearly one-hot.  The output is then close to
    one dequantised V row, whose bf16 rounding alone averages about 1.5e-3,
    so the check takes the output in float32 against the kernel's arithmetic
    bound (see _decode_only_check)."""
    cfg = workloads.DecodeConfig("p", 4, 8, 2, 128, 16, 0, 3000, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=58, ctx=[100, 1100, 2100, 3000])
    d.q = (d.q.float() * gain).to(torch.bfloat16)
    _decode_only_check(d, d.scale, f"peaked gain={gain}")


@pytest.mark.parametrize("G", [2, 4])
def test_q8_decode_wide_scales(G):
    """Key and value scales spread over 2^-6..2^6 and 2^-13..2^13 of the usual
    range, some all-zero value rows, and random codes with NaN scales in the
    unfilled slots: the value scale rides in the softmax weight, so the fp16
    weights must not lose the small-scale tokens nor overflow on the large."""
    Hkv = 2
    cfg = workloads.DecodeConfig("w", 6, G * Hkv, Hkv, 128, 16, 0, 3000, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=54, ctx=[1, 17, 700, 1024, 2049, 3000])
    gen = torch.Generator().manual_seed(55)
    filled = ~torch.isnan(d.k_scale)
    d.k_scale[filled] *= torch.exp2(torch.empty(int(filled.sum())).uniform_(-6, 6, generator=gen))
    d.v_scale[filled] *= torch.exp2(torch.empty(int(filled.sum())).uniform_(-13, 13, generator=gen))
    zero = filled & (torch.rand(d.v_scale.shape, generator=gen) < 0.05)
    d.v_scale[zero] = 0.0
    hole = ~filled
    junk = torch.randint(-128, 128, d.kq_cache.shape, generator=gen, dtype=torch.int32).to(torch.int8)
    d.kq_cache[hole] = junk[hole]
    d.vq_cache[hole] = junk.flip(0)[hole]
    _decode_only_check(d, d.scale, f"wide scales G={G}")


def test_q8_decode_query_beyond_fp16_range():
    """Query elements up to 1e5 (past fp16's 65504) with a small softmax
    scale: the tensor-core decode takes q in fp16 after an exact power-of-two
    prescale, which must leave the result unchanged."""
    Hkv, G = 2, 4
    cfg = workloads.DecodeConfig("b", 4, G * Hkv, Hkv, 128, 16, 0, 1200, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=56, ctx=[5, 300, 1024, 1200])
    q = d.q.float()
    q[:, :, 3] = 1.0e5
    q[0, 1, 7] = -7.0e4
    d.q = q.to(torch.bfloat16)
    _decode_only_check(d, 2.0e-6, "large q")


def test_q8_decode_empty_context_and_bad_block():
    """An empty context gives out = 0 and lse = -inf; a table entry outside
    the cache is reported (status 5) and skipped without a fault."""
    cfg = workloads.DecodeConfig("e", 3, 8, 2, 128, 16, 0, 200, 2)
    d = workloads.make_decode_inputs_q8(cfg, seed=58, ctx=[10, 100, 200])
    g = _dev(d)
    lens = g["ctx"].clone()
    lens[0] = 0
    ws = lib.Workspace(lib.paged_decode_workspace_size(3, 8, d.block_table.shape[1], 16, 128))
    out, lse = lib.paged_decode_attn_q8(g["q"], g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"],
                                        g["block_table"], lens, d.scale, return_lse=True, workspace=ws)
    assert ws.status() == 0
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    lens_cpu = lens.cpu()
    ro, rl = oracle.paged_decode_q8(d.q[1:], d.kq_cache.numpy(), d.vq_cache.numpy(), d.k_scale.numpy(),
                                    d.v_scale.numpy(), d.block_table[1:], lens_cpu[1:], d.scale)
    assert_out_close(out[1:], ro)
    assert_lse_close(lse[1:], rl)
    bt = g["block_table"].clone()
    bt[2, 3] = -7
    ws.reset()
    lib.paged_decode_attn_q8(g["q"], g["kq_cache"], g["vq_cache"], g["k_scale"], g["v_scale"], bt, lens, d.scale,
                             workspace=ws)
    assert ws.status() == 5


def test_q8_decode_subnormal_value_weights():
    """One 16-token block whose top-scoring token has value scale 0 and whose
    other tokens score 125 log2 units lower: every value weight p * vs of the
    block is subnormal.  The value-weight reference must not be set from
    such a block (1 / ref would overflow and 0 * inf poison the output); the
    result is finite and matches the oracle (whose output is ~1e-40 here)."""
    cfg = workloads.DecodeConfig("t", 1, 4, 1, 128, 16, 0, 16, 2)
    d = workloads.make_decode_inputs_q8(cfg, seed=59, ctx=[16])
    blk = int(d.block_table[0, 0])
    d.kq_cache[blk, 0] = 0
    d.kq_cache[blk, 0, 0, 0] = 127          # token 0: the only non-zero key
    d.k_scale[blk, 0] = 0.01
    d.k_scale[blk, 0, 0] = 125.0 / (127 * d.scale * 1.4426950408889634)  # score 125 (log2) above the rest
    d.v_scale[blk, 0] = 0.01
    d.v_scale[blk, 0, 0] = 0.0              # the top token's value row is zero
    q = torch.zeros_like(d.q.float())
    q[0, :, 0] = 1.0
    d.q = q.to(torch.bfloat16)
    # weights p * vs below 1e-30 are dropped (each token then moves the output
    # by at most 1e-30 * 127 / l, l >= 1): a floor far below anything visible
    _decode_only_check(d, d.scale, "subnormal value weights", abs_floor=1e-20)


def _fused_check(d, note=""):
    """paged_decode_attn_append_q8 against the oracle (its append, then its
    decode over the dequantised cache) and, bit for bit, against the two
    separate calls on a copy of the same cache."""
    g = _dev(d)
    ws = lib.Workspace(lib.paged_decode_workspace_size(d.cfg.B, d.cfg.Hq, d.block_table.shape[1], 16, d.cfg.D))
    out, lse = lib.paged_decode_attn_append_q8(g["q"], g["k_new"], g["v_new"], g["kq_cache"], g["vq_cache"],
                                               g["k_scale"], g["v_scale"], g["block_table"], g["pos"], d.scale,
                                               return_lse=True, workspace=ws)
    assert ws.status() == 0
    kq, vq, ks, vs = oracle.kv_append_q8(d.kq_cache, d.vq_cache, d.k_scale, d.v_scale, d.block_table, d.pos,
                                         d.k_new, d.v_new)
    np.testing.assert_array_equal(g["kq_cache"].cpu().numpy(), kq)
    np.testing.assert_array_equal(g["vq_cache"].cpu().numpy(), vq)
    np.testing.assert_array_equal(g["k_scale"].cpu().numpy().view(np.int32), ks.view(np.int32))
    np.testing.assert_array_equal(g["v_scale"].cpu().numpy().view(np.int32), vs.view(np.int32))
    ro, rl = oracle.paged_decode_q8(d.q, kq, vq, ks, vs, d.block_table, d.ctx_lens, d.scale)
    assert_out_close(out, ro, what="q8 fused out" + note)
    assert_lse_close(lse, rl, what="q8 fused lse" + note)
    h = _dev(d)
    lib.kv_append_q8(h["kq_cache"], h["vq_cache"], h["k_scale"], h["v_scale"], h["block_table"], h["pos"],
                     h["k_new"], h["v_new"], workspace=ws)
    o2, l2 = lib.paged_decode_attn_q8(h["q"], h["kq_cache"], h["vq_cache"], h["k_scale"], h["v_scale"],
                                      h["block_table"], h["ctx_lens"], d.scale, return_lse=True, workspace=ws)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("D,G", [(128, 4), (128, 1), (128, 8), (64, 4)])
def test_q8_fused_append_decode_small(D, G):
    """Contexts that put the new token at block and split edges (0, 15, 16,
    1023, 1024 tokens before it); D = 64 runs the append kernel first."""
    Hkv = 2
    cfg = workloads.DecodeConfig("f", 9, G * Hkv, Hkv, D, 16, 0, 1500, 4)
    d = workloads.make_decode_inputs_q8(cfg, seed=61, ctx=[0, 15, 16, 511, 512, 1023, 1024, 1300, 1500])
    _fused_check(d, f" D={D} G={G}")


def test_q8_fused_append_decode_full_workload():
    d = workloads.make_decode_inputs_q8(workloads.DECODE_CONFIGS["decode"], seed=0)
    _fused_check(d, " full")


def test_q8_fused_idle_and_bad_positions():
    """pos < 0 is an idle sequence (nothing written, out = 0, lse = -inf); a
    position past the table is reported (status 5) with nothing written."""
    cfg = workloads.DecodeConfig("q", 4, 8, 2, 128, 16, 0, 100, 2)
    d = workloads.make_decode_inputs_q8(cfg, seed=62, ctx=[3, 30, 60, 90])
    g = _dev(d)
    pos = g["pos"].clone()
    pos[1] = -1
    pos[2] = 16 * d.block_table.shape[1]
    ws = lib.Workspace(lib.paged_decode_workspace_size(4, 8, d.block_table.shape[1], 16, 128))
    out, lse = lib.paged_decode_attn_append_q8(g["q"], g["k_new"], g["v_new"], g["kq_cache"], g["vq_cache"],
                                               g["k_scale"], g["v_scale"], g["block_table"], pos, d.scale,
                                               return_lse=True, workspace=ws)
    assert ws.status() == 5
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    p2 = d.pos.clone()
    p2[1] = -1
    p2[2] = -1
    kq, vq, ks, vs = oracle.kv_append_q8(d.kq_cache, d.vq_cache, d.k_scale, d.v_scale, d.block_table, p2,
                                         d.k_new, d.v_new)
    np.testing.assert_array_equal(g["kq_cache"].cpu().numpy(), kq)
    np.testing.assert_array_equal(g["vq_cache"].cpu().numpy(), vq)
    np.testing.assert_array_equal(g["k_scale"].cpu().numpy().view(np.int32), ks.view(np.int32))
    np.testing.assert_array_equal(g["v_scale"].cpu().numpy().view(np.int32), vs.view(np.int32))
    sel = [0, 3]
    ro, rl = oracle.paged_decode_q8(d.q[sel], kq, vq, ks, vs, d.block_table[sel], d.ctx_lens[sel], d.scale)
    assert_out_close(out[sel], ro, what="q8 fused out, live sequences")
    assert_lse_close(lse[sel], rl, what="q8 fused lse, live sequences")
