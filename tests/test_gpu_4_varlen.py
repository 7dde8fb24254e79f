"""GPU parity of the key-length form of masked attention (attn_fwd_varlen)
and of the boolean key_padding_mask converter.

attn_fwd_varlen(key_lens) must equal the oracle with the additive mask
0 for keys < key_lens[b] and -inf after (the padded-tail form of the first
page), including lengths 0, 1, one tile, one past a tile, and all keys."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 64), (torch.bfloat16, 128), (torch.float32, 64)])
def test_varlen_matches_the_equivalent_padding_mask(dtype, D):
    lens = [0, 1, 127, 128, 129, 300, 517]
    B, Pk = len(lens), 517
    inp = workloads.make_attn(B, 4, 2, 200, Pk, D, dtype=dtype, n_pad=[Pk - n for n in lens], seed=31)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = lib.Workspace(256)
    o, l = lib.attn_fwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), kl, inp.scale, workspace=ws)
    assert ws.status() == 0
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)  # mask = the padded tails
    fp32 = dtype == torch.float32
    assert_out_close(o, ro, fp32_inputs=fp32)
    assert_lse_close(l, rl)
    # and the same as attn_fwd with the additive mask, call for call
    o2, l2 = lib.attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.mask.cuda(), inp.scale)
    np.testing.assert_allclose(o.float().cpu().numpy(), o2.float().cpu().numpy(), atol=2e-2)


def test_varlen_clamps_lengths():
    inp = workloads.make_attn(2, 2, 2, 50, 100, 64, dtype=torch.bfloat16, with_mask=False, seed=32)
    kl = torch.tensor([-5, 1000], dtype=torch.int32, device="cuda")
    o, l = lib.attn_fwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), kl, inp.scale)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(l[0]))
    ro, rl = oracle.attn(inp.q[1:], inp.k[1:], inp.v[1:], None, inp.scale)
    assert_out_close(o[1:], ro)
    assert_lse_close(l[1:], rl)


def test_key_padding_mask_conversion_and_direction():
    """True in a key_padding_mask means 'ignore this key' (first page, note on
    the mask direction); the converter yields -inf there and 0 elsewhere, and
    attention with it equals dropping those keys."""
    g = torch.Generator().manual_seed(33)
    kpm = torch.rand(3, 300, generator=g) < 0.3
    add = lib.key_padding_to_additive(kpm.cuda()).cpu()
    assert torch.equal(torch.isneginf(add), kpm) and torch.all(add[~kpm] == 0)
    inp = workloads.make_attn(3, 2, 2, 40, 300, 64, dtype=torch.bfloat16, with_mask=False, seed=34)
    o, _ = lib.attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), add.cuda(), inp.scale)
    ro, _ = oracle.attn(inp.q, inp.k, inp.v, add, inp.scale)
    assert_out_close(o, ro)
    # the inverted convention (True = keep) gives a clearly different answer
    inv = lib.key_padding_to_additive((~kpm).cuda())
    o_inv, _ = lib.attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inv, inp.scale)
    assert (o_inv.float() - o.float()).abs().max().item() > 0.1


@pytest.mark.parametrize("D,out_dtype,with_lse", [(64, torch.bfloat16, True), (128, torch.float32, False)])
def test_varlen_with_a_split_last_wave(D, out_dtype, with_lse):
    """160 heads: the units of the last wave are split over their key tiles;
    per-batch key lengths then bound each part's tiles.  f32 output and no
    LSE buffer go through the same merge."""
    lens = [700, 129]
    B, Pk = 2, 700
    inp = workloads.make_attn(B, 80, 16, 230, Pk, D, dtype=torch.bfloat16, n_pad=[Pk - n for n in lens], seed=35)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = lib.Workspace(lib.attn_fwd_workspace_size_for(B, 16, Pk, D))
    out = torch.empty(inp.q.shape, dtype=out_dtype, device="cuda")
    res = lib.attn_fwd_varlen(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), kl, inp.scale, out=out, workspace=ws,
                              return_lse=with_lse)
    assert ws.status() == 0
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(out, ro, fp32_inputs=False)
    if with_lse:
        assert_lse_close(res[1], rl)
