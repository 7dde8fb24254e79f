"""GPU parity of the paged-cache calls against the oracle: kv_append and the
block-table gather bit for bit, paged GQA decode within the bf16 tolerances,
at small ragged sizes and at the full decode workload (64 sequences, 32 query
heads over 8 KV heads, D 128, contexts uniform in [512, 8192])."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(d: workloads.DecodeInputs):
    return {k: getattr(d, k).to(DEV) for k in ("k_cache", "v_cache", "block_table", "pos", "ctx_lens", "ctx",
                                               "k_new", "v_new", "q")}


SMALL = workloads.DecodeConfig("small", 7, 8, 2, 128, 16, 0, 1100, 5)


@pytest.mark.parametrize("D,ctx", [(128, [0, 1, 15, 16, 17, 511, 512]), (64, [3, 31, 32, 33, 700, 1023, 1100])])
def test_kv_append_bit_exact(D, ctx):
    cfg = workloads.DecodeConfig("a", len(ctx), 8, 2, D, 16, 0, 1100, 5)
    d = workloads.make_decode_inputs(cfg, seed=3, ctx=ctx)
    g = _dev(d)
    ws = lib.Workspace(256)
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"], workspace=ws)
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    # NaN sentinels compare as bits, so untouched slots must keep their exact pattern
    assert np.array_equal(g["k_cache"].cpu().view(torch.int16).numpy(), ek)
    assert np.array_equal(g["v_cache"].cpu().view(torch.int16).numpy(), ev)
    assert ws.status() == 0


def test_kv_append_skips_idle_and_flags_bad_positions():
    d = workloads.make_decode_inputs(SMALL, seed=4, ctx=[5, 6, 7, 8, 9, 10, 11])
    g = _dev(d)
    pos = g["pos"].clone()
    pos[1] = -1  # idle sequence: nothing written
    pos[2] = 16 * d.block_table.shape[1]  # past the table
    ws = lib.Workspace(256)
    before = g["k_cache"].clone()
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], pos, g["k_new"], g["v_new"], workspace=ws)
    assert ws.status() == 5  # ATTN_ERR_DEVICE_BOUNDS
    p2 = pos.cpu().clone()
    p2[1] = d.pos[1]
    p2[2] = d.pos[2]
    exp_k, _ = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    got = g["k_cache"].cpu().view(torch.int16).numpy()
    for b in range(7):
        blk = int(d.block_table[b, int(d.pos[b]) // 16])
        slot = int(d.pos[b]) % 16
        if b in (1, 2):
            assert np.array_equal(got[blk, :, slot], before.cpu().view(torch.int16).numpy()[blk, :, slot])
        else:
            assert np.array_equal(got[blk, :, slot], exp_k[blk, :, slot])


@pytest.mark.parametrize("D", [64, 128])
def test_paged_gather_bit_exact(D):
    cfg = workloads.DecodeConfig("g", 5, 8, 4, D, 16, 1, 900, 3)
    d = workloads.make_decode_inputs(cfg, seed=5, ctx=[1, 16, 17, 512, 900])
    g = _dev(d)
    max_len = int(d.ctx.max())
    got = lib.paged_kv_gather(g["k_cache"], g["block_table"], g["ctx"], max_len)
    exp = oracle.paged_gather(d.k_cache, d.block_table, d.ctx)
    got_bits = got.cpu().view(torch.int16).numpy()
    for b in range(5):
        L = int(d.ctx[b])
        assert np.array_equal(got_bits[b, :, :L], exp[b])
        assert np.all(got_bits[b, :, L:] == 0)


def test_gather_flags_bad_block_ids():
    d = workloads.make_decode_inputs(SMALL, seed=6, ctx=[40] * 7)
    g = _dev(d)
    bt = g["block_table"].clone()
    bt[3, 1] = d.num_blocks + 5
    ws = lib.Workspace(256)
    lib.paged_kv_gather(g["k_cache"], bt, g["ctx"], 40, workspace=ws)
    assert ws.status() == 5


def _decode_and_check(d: workloads.DecodeInputs, seed_note=""):
    g = _dev(d)
    ws = lib.Workspace(lib.paged_decode_workspace_size(d.cfg.B, d.cfg.Hq, d.block_table.shape[1], 16, d.cfg.D))
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"], workspace=ws)
    out, lse = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], d.scale,
                                     return_lse=True, workspace=ws)
    assert ws.status() == 0
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    ro, rl = oracle.paged_decode(d.q, torch.from_numpy(ek).view(torch.bfloat16),
                                 torch.from_numpy(ev).view(torch.bfloat16), d.block_table, d.ctx_lens, d.scale)
    assert_out_close(out, ro, what="decode out" + seed_note)
    assert_lse_close(lse, rl, what="decode lse" + seed_note)
    return out


@pytest.mark.parametrize("D,G", [(128, 4), (128, 1), (128, 2), (128, 8), (64, 4), (64, 2), (64, 1), (64, 8)])
def test_paged_decode_small(D, G):
    Hkv = 2
    cfg = workloads.DecodeConfig("s", 9, G * Hkv, Hkv, D, 16, 0, 1500, 4)
    # L = ctx + 1: 1 token, a full block, one past a block, a whole split, one
    # past a split, several splits with a ragged tail
    d = workloads.make_decode_inputs(cfg, seed=7, ctx=[0, 15, 16, 511, 512, 1023, 1024, 1300, 1500])
    _decode_and_check(d, f" D={D} G={G}")


def test_paged_decode_long_context():
    """Contexts of 40,000 and 33,000 tokens: 40 and 33 splits of 1024, more
    than the 32 the split merge takes in one pass."""
    cfg = workloads.DecodeConfig("l", 3, 8, 2, 128, 16, 0, 40000, 4)
    d = workloads.make_decode_inputs(cfg, seed=19, ctx=[40000, 33000, 100])
    _decode_and_check(d, " long")


@pytest.mark.parametrize("D", [128, 64])
def test_paged_decode_reuses_its_workspace(D):
    """Three decode calls through one workspace with different context
    lengths (so each sequence has a different number of splits every time):
    each call's split counts start afresh under its own generation, and every
    call matches the oracle."""
    cfg = workloads.DecodeConfig("w", 5, 8, 2, D, 16, 0, 3000, 4)
    d = workloads.make_decode_inputs(cfg, seed=89, ctx=[3000, 2500, 1024, 700, 5])
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    kc, vc = torch.from_numpy(ek).view(torch.bfloat16), torch.from_numpy(ev).view(torch.bfloat16)
    g = {k: getattr(d, k).to(DEV) for k in ("block_table", "q")}
    gk, gv = kc.to(DEV), vc.to(DEV)
    ws = lib.Workspace(lib.paged_decode_workspace_size(cfg.B, cfg.Hq, d.block_table.shape[1], 16, D))
    full = d.ctx_lens.clone()
    for lens in (full, torch.clamp(full - 1100, min=0), torch.tensor([1, 1025, 2049, 3001, 0], dtype=torch.int32)):
        lens = torch.minimum(lens.to(torch.int32), full)
        out, lse = lib.paged_decode_attn(g["q"], gk, gv, g["block_table"], lens.to(DEV), d.scale, return_lse=True,
                                         workspace=ws)
        assert ws.status() == 0
        ro, rl = oracle.paged_decode(d.q, kc, vc, d.block_table, lens, d.scale)
        assert_out_close(out, ro, what=f"reused workspace, lens {lens.tolist()}")
        assert_lse_close(lse, rl)


def test_paged_decode_workspace_contents_do_not_matter():
    """The split counts carry each call's generation, so a decode workspace
    needs no clearing: filled with 0x7F bytes, with random bytes, or left
    with the partials of a call of another shape (a larger batch, longer
    contexts), it gives the oracle's result each time (only the status word
    is reset)."""
    cfg = workloads.DecodeConfig("z", 3, 8, 2, 128, 16, 0, 2100, 4)
    d = workloads.make_decode_inputs(cfg, seed=90, ctx=[2100, 900, 40])
    big = workloads.make_decode_inputs(workloads.DecodeConfig("zb", 9, 16, 2, 128, 16, 0, 4000, 4), seed=91,
                                       ctx=[4000, 3900, 10, 2048, 1025, 3000, 5, 1, 2500])

    def run(inp, ws):
        ek, ev = oracle.kv_append(inp.k_cache, inp.v_cache, inp.block_table, inp.pos, inp.k_new, inp.v_new)
        kc, vc = torch.from_numpy(ek).view(torch.bfloat16), torch.from_numpy(ev).view(torch.bfloat16)
        out = lib.paged_decode_attn(inp.q.to(DEV), kc.to(DEV), vc.to(DEV), inp.block_table.to(DEV),
                                    inp.ctx_lens.to(DEV), inp.scale, workspace=ws)
        assert ws.status() == 0
        ro, _ = oracle.paged_decode(inp.q, kc, vc, inp.block_table, inp.ctx_lens, inp.scale)
        assert_out_close(out, ro, what=f"decode {inp.cfg.name}")

    need = max(lib.paged_decode_workspace_size(x.cfg.B, x.cfg.Hq, x.block_table.shape[1], 16, 128) for x in (d, big))
    ws = lib.Workspace(need)
    ws.tensor.fill_(0x7F)
    ws.reset()
    run(d, ws)
    g = torch.Generator(device="cpu").manual_seed(92)
    ws.tensor.copy_(torch.randint(0, 256, ws.tensor.shape, generator=g, dtype=torch.uint8))
    ws.reset()
    run(d, ws)
    run(big, ws)  # another shape: its partials now lie where the small call keeps its counts
    run(d, ws)
    run(big, ws)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("gain", [8.0, 40.0])
def test_paged_decode_peaked_scores(D, gain):
    """Queries scaled up so that the scores spread over tens to hundreds of
    log2 units: the running maximum moves within blocks, across the warps of
    a split and across splits, and the weights are nearly one-hot."""
    cfg = workloads.DecodeConfig("p", 4, 8, 2, D, 16, 0, 3000, 4)
    d = workloads.make_decode_inputs(cfg, seed=87, ctx=[100, 1100, 2100, 3000])
    d.q = (d.q.float() * gain).to(torch.bfloat16)
    _decode_and_check(d, f" D={D} gain={gain}")


def test_paged_decode_f32_output_and_strided_q():
    cfg = workloads.DecodeConfig("s", 3, 8, 2, 128, 16, 100, 600, 2)
    d = workloads.make_decode_inputs(cfg, seed=8)
    g = _dev(d)
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"])
    # q as a strided view (heads of a wider buffer)
    qbuf = torch.zeros(3, 16, 128, dtype=torch.bfloat16, device=DEV)
    qbuf[:, ::2] = g["q"]
    qv = qbuf[:, ::2]
    out = torch.empty(3, 8, 128, dtype=torch.float32, device=DEV)
    lib.paged_decode_attn(qv, g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], d.scale, out=out)
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    ro, _ = oracle.paged_decode(d.q, torch.from_numpy(ek).view(torch.bfloat16),
                                torch.from_numpy(ev).view(torch.bfloat16), d.block_table, d.ctx_lens, d.scale)
    assert_out_close(out, ro, what="decode f32 out")


def test_paged_decode_empty_context_and_bad_block():
    cfg = workloads.DecodeConfig("e", 3, 8, 2, 128, 16, 0, 200, 2)
    d = workloads.make_decode_inputs(cfg, seed=9, ctx=[10, 100, 200])
    g = _dev(d)
    lens = g["ctx"].clone()
    lens[0] = 0  # no tokens at all
    ws = lib.Workspace(lib.paged_decode_workspace_size(3, 8, d.block_table.shape[1], 16, 128))
    out, lse = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], lens, d.scale,
                                     return_lse=True, workspace=ws)
    assert ws.status() == 0
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    lens_cpu = lens.cpu()
    ro, rl = oracle.paged_decode(d.q[1:], d.k_cache, d.v_cache, d.block_table[1:], lens_cpu[1:], d.scale)
    assert_out_close(out[1:], ro)
    assert_lse_close(lse[1:], rl)
    # a table entry outside the cache is reported, and the call neither faults nor hangs
    bt = g["block_table"].clone()
    bt[2, 3] = -7
    ws.reset()
    lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], bt, lens, d.scale, workspace=ws)
    assert ws.status() == 5


def test_paged_decode_full_workload():
    """64 sequences x 32 query heads, KV heads 8, D 128, contexts U[512, 8192]:
    append then decode, every output against the oracle."""
    d = workloads.make_decode_inputs(workloads.DECODE_CONFIGS["decode"], seed=0)
    _decode_and_check(d, " full")


def test_incremental_decode_equals_recompute_on_gpu():
    """The decode of the appended token equals the last row of full attention
    over the gathered contiguous sequence, both computed on the GPU
    (paged_decode_attn vs attn_fwd over paged_kv_gather output)."""
    cfg = workloads.DecodeConfig("r", 4, 8, 2, 128, 16, 300, 900, 2)
    d = workloads.make_decode_inputs(cfg, seed=10)
    g = _dev(d)
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"])
    out, lse = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], d.scale,
                                     return_lse=True)
    Lmax = int(d.ctx_lens.max())
    kcont = lib.paged_kv_gather(g["k_cache"], g["block_table"], g["ctx_lens"], Lmax)
    vcont = lib.paged_kv_gather(g["v_cache"], g["block_table"], g["ctx_lens"], Lmax)
    for b in range(4):
        L = int(d.ctx_lens[b])
        o2, l2 = lib.attn_fwd(g["q"][b:b + 1].unsqueeze(2).contiguous(), kcont[b:b + 1, :, :L].contiguous(),
                              vcont[b:b + 1, :, :L].contiguous(), None, d.scale)
        diff = (o2[0, :, 0].float() - out[b].float()).abs().max().item()
        assert diff <= 2e-2
        assert (l2[0, :, 0] - lse[b]).abs().max().item() <= 1e-3


def _fused_and_check(d: workloads.DecodeInputs, note=""):
    """paged_decode_attn_append against the oracle's kv_append then decode:
    the cache bit for bit, the outputs within the bf16 tolerances."""
    g = _dev(d)
    ws = lib.Workspace(lib.paged_decode_workspace_size(d.cfg.B, d.cfg.Hq, d.block_table.shape[1], 16, d.cfg.D))
    out, lse = lib.paged_decode_attn_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"],
                                            g["block_table"], g["pos"], d.scale, return_lse=True, workspace=ws)
    assert ws.status() == 0
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table, d.pos, d.k_new, d.v_new)
    assert np.array_equal(g["k_cache"].cpu().view(torch.int16).numpy(), ek)
    assert np.array_equal(g["v_cache"].cpu().view(torch.int16).numpy(), ev)
    ro, rl = oracle.paged_decode(d.q, torch.from_numpy(ek).view(torch.bfloat16),
                                 torch.from_numpy(ev).view(torch.bfloat16), d.block_table, d.ctx_lens, d.scale)
    assert_out_close(out, ro, what="fused decode out" + note)
    assert_lse_close(lse, rl, what="fused decode lse" + note)
    return out, lse


@pytest.mark.parametrize("D,G", [(128, 4), (128, 8), (64, 2), (64, 1)])
def test_fused_append_decode_small(D, G):
    """The new token's slot holds NaN before the call: reading it instead of
    the substituted row would show in every output of that sequence."""
    Hkv = 2
    cfg = workloads.DecodeConfig("f", 9, G * Hkv, Hkv, D, 16, 0, 1500, 4)
    d = workloads.make_decode_inputs(cfg, seed=17, ctx=[0, 15, 16, 511, 512, 1023, 1024, 1300, 1500])
    _fused_and_check(d, f" D={D} G={G}")


def test_fused_append_decode_full_workload():
    d = workloads.make_decode_inputs(workloads.DECODE_CONFIGS["decode"], seed=0)
    out, lse = _fused_and_check(d, " full")
    # and the same numbers as the two-launch path on the same inputs
    g = _dev(d)
    lib.kv_append(g["k_cache"], g["v_cache"], g["block_table"], g["pos"], g["k_new"], g["v_new"])
    o2, l2 = lib.paged_decode_attn(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["ctx_lens"], d.scale,
                                   return_lse=True)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_fused_append_idle_and_out_of_table_positions():
    d = workloads.make_decode_inputs(SMALL, seed=18, ctx=[5, 6, 7, 8, 9, 10, 11])
    g = _dev(d)
    pos = g["pos"].clone()
    pos[1] = -1  # idle: cache untouched, empty result
    pos[2] = 16 * d.block_table.shape[1]  # past the table: reported, cache untouched
    before = g["k_cache"].cpu().view(torch.int16).numpy().copy()
    ws = lib.Workspace(lib.paged_decode_workspace_size(7, 8, d.block_table.shape[1], 16, 128))
    out, lse = lib.paged_decode_attn_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"],
                                            g["block_table"], pos, d.scale, return_lse=True, workspace=ws)
    assert ws.status() == 5
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    got = g["k_cache"].cpu().view(torch.int16).numpy()
    for b in (1, 2):
        p = int(d.pos[b])
        blk, slot = int(d.block_table[b, p // 16]), p % 16
        assert np.array_equal(got[blk, :, slot], before[blk, :, slot])
    keep = [0, 3, 4, 5, 6]
    ek, ev = oracle.kv_append(d.k_cache, d.v_cache, d.block_table[keep], d.pos[keep], d.k_new[keep], d.v_new[keep])
    ro, rl = oracle.paged_decode(d.q[keep], torch.from_numpy(ek).view(torch.bfloat16),
                                 torch.from_numpy(ev).view(torch.bfloat16), d.block_table[keep], d.ctx_lens[keep],
                                 d.scale)
    assert_out_close(out[keep], ro)
    assert_lse_close(lse[keep], rl)
