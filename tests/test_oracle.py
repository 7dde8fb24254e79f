"""Pins for the CPU oracle (runs without a GPU).

Each test checks the oracle against something other than itself: brute force
in 60-digit arithmetic, PyTorch's own fp64 scaled_dot_product_attention and
logsumexp (library routines), closed forms, invariants the pages state, and
the numbers the pages print.  Each is chosen so that a plausible slip in the
oracle (a dropped mask term, a scaled mask, log base 2 instead of e, a
transposed operand, a wrong GQA head map, a wrong block/slot split, an
unstable merge) fails at least one of them; ``test_planted_mistakes`` plants
several such slips in a copy of the oracle and checks that they are caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# helpers that are NOT the oracle
# --------------------------------------------------------------------------
def _mp_attention(q, k, v, mask, scale, group):
    """Brute force in 60-digit arithmetic, without the max shift: every
    probability is exp(s_j) / sum_k exp(s_k) evaluated directly."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    B, Hq, Pq, D = q.shape
    Pk = k.shape[2]
    out = np.zeros((B, Hq, Pq, D))
    lse = np.zeros((B, Hq, Pq))
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(Pq):
                s = []
                for j in range(Pk):
                    if mask is not None and math.isinf(float(mask[b, j])):
                        s.append(None)
                        continue
                    dot = mpmath.fsum(mpmath.mpf(float(q[b, h, i, d])) * mpmath.mpf(float(k[b, g, j, d]))
                                      for d in range(D))
                    add = mpmath.mpf(float(mask[b, j])) if mask is not None else 0
                    s.append(mpmath.mpf(scale) * dot + add)
                e = [mpmath.e ** x if x is not None else mpmath.mpf(0) for x in s]
                z = mpmath.fsum(e)
                if z == 0:
                    lse[b, h, i] = -math.inf
                    continue
                lse[b, h, i] = float(mpmath.log(z))
                for d in range(D):
                    out[b, h, i, d] = float(mpmath.fsum(e[j] * mpmath.mpf(float(v[b, g, j, d]))
                                                         for j in range(Pk)) / z)
    return out, lse


def _sdpa_f64(q, k, v, mask, scale):
    """PyTorch's fp64 CPU SDPA with an additive float mask, plus logsumexp."""
    q64, k64, v64 = (t.to(torch.float64) for t in (q, k, v))
    group = q.shape[1] // k.shape[1]
    k64 = k64.repeat_interleave(group, dim=1)
    v64 = v64.repeat_interleave(group, dim=1)
    am = None
    if mask is not None:
        am = mask.to(torch.float64)[:, None, None, :]
    out = F.scaled_dot_product_attention(q64, k64, v64, attn_mask=am, scale=scale)
    logits = torch.matmul(q64, k64.transpose(-1, -2)) * scale
    if am is not None:
        logits = logits + am
    lse = torch.logsumexp(logits, dim=-1)
    return out.numpy(), lse.numpy()


# --------------------------------------------------------------------------
# attention definition
# --------------------------------------------------------------------------
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (3, 1)])
def test_attn_brute_force_60_digits(Hq, Hkv):
    inp = workloads.make_attn(1, Hq, Hkv, 3, 6, 4, dtype=torch.float32, n_pad=2, seed=11)
    inp.mask[0, 1] = float("-inf")  # an interior masked key as well
    inp.mask[0, 0] = 0.75  # a finite additive mask value
    out, lse = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.37)
    ref_o, ref_l = _mp_attention(inp.q, inp.k, inp.v, inp.mask, 0.37, Hq // Hkv)
    np.testing.assert_allclose(out, ref_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,Hq,Hkv,Pq,Pk,D,pad", [
    (1, 2, 2, 33, 47, 16, 5),
    (2, 4, 1, 17, 130, 64, [0, 129]),
    (1, 3, 3, 1, 1, 8, 0),
    (2, 8, 2, 40, 200, 128, [7, 64]),
])
def test_attn_matches_library_sdpa(dtype, B, Hq, Hkv, Pq, Pk, D, pad):
    inp = workloads.make_attn(B, Hq, Hkv, Pq, Pk, D, dtype=dtype, n_pad=pad, seed=3)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.attn(inp.q, inp.k, inp.v, inp.mask, scale)
    ref_o, ref_l = _sdpa_f64(inp.q, inp.k, inp.v, inp.mask, scale)
    np.testing.assert_allclose(out, ref_o, rtol=1e-11, atol=1e-12)
    # PyTorch's fp64 CPU logits/logsumexp were seen, now and then, to come out
    # ~1.4e-10 relative off (against an exact-sum reference, while the oracle
    # stayed within 1e-15); the 60-digit brute-force pins hold the oracle to 1e-12
    np.testing.assert_allclose(lse, ref_l, rtol=1e-9, atol=1e-9)


def test_attn_packed_strides_match_contiguous():
    """The packed [T, H, D] layout (ring-attention page, forward_ring_kv_chunk)
    is the same attention as the contiguous [1, H, T, D] copy."""
    cfg = workloads.AttnConfig("p", 1, 4, 4, 70, 70, 32, torch.bfloat16, packed=True)
    inp = workloads.make_attn_inputs(cfg, seed=5)
    assert not inp.q.is_contiguous()
    a = oracle.attn(inp.q, inp.k, inp.v, None, 0.2)
    b = oracle.attn(inp.q.contiguous(), inp.k.contiguous(), inp.v.contiguous(), None, 0.2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_attn_row_subset_matches_full():
    inp = workloads.make_attn(2, 4, 2, 21, 50, 16, dtype=torch.bfloat16, n_pad=[3, 9], seed=8)
    full_o, full_l = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.25)
    rows = [0, 5, 83, 84, 167, 100]
    o, l = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.25, rows=rows)
    flat_o = full_o.reshape(-1, 16)
    np.testing.assert_array_equal(o, flat_o[rows])
    np.testing.assert_array_equal(l, full_l.reshape(-1)[rows])


def test_equal_scores_give_mean_of_unmasked_values():
    """Closed form: with q = 0 every score is equal, so each output row is the
    mean of the unmasked V rows and lse = ln(number of unmasked keys)."""
    inp = workloads.make_attn(2, 4, 4, 9, 77, 32, dtype=torch.float32, n_pad=[13, 0], seed=1)
    q = torch.zeros_like(inp.q)
    out, lse = oracle.attn(q, inp.k, inp.v, inp.mask, 0.125)
    for b, n_pad in enumerate([13, 0]):
        n = 77 - n_pad
        mean = inp.v[b, :, :n, :].to(torch.float64).mean(dim=1).numpy()  # [H, D]
        for i in range(9):
            np.testing.assert_allclose(out[b, :, i, :], mean, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(lse[b], math.log(n), rtol=0, atol=1e-13)


def test_single_unmasked_key_returns_its_value_row():
    """Masking every key but j returns exactly v_j, with lse = the lone score."""
    inp = workloads.make_attn(1, 2, 2, 5, 40, 16, dtype=torch.bfloat16, seed=2)
    j = 23
    mask = torch.full((1, 40), float("-inf"))
    mask[0, j] = 0.0
    out, lse = oracle.attn(inp.q, inp.k, inp.v, mask, 0.3)
    v = inp.v.to(torch.float64).numpy()
    q = inp.q.to(torch.float64).numpy()
    k = inp.k.to(torch.float64).numpy()
    for h in range(2):
        for i in range(5):
            np.testing.assert_array_equal(out[0, h, i], v[0, h, j])
            s = 0.3 * float(np.dot(q[0, h, i], k[0, h, j]))
            assert abs(lse[0, h, i] - s) < 1e-12


def test_mask_direction_matters():
    """key_padding_mask True means 'ignore' while SDPA's bool mask True means
    'participate' (first page, mask-direction note): feeding the complement
    must change the result; the additive form used here is unambiguous."""
    inp = workloads.make_attn(1, 2, 2, 8, 64, 16, dtype=torch.float32, n_pad=20, seed=4)
    inverted = torch.where(torch.isinf(inp.mask), torch.zeros_like(inp.mask),
                           torch.full_like(inp.mask, float("-inf")))
    a, _ = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.25)
    b, _ = oracle.attn(inp.q, inp.k, inp.v, inverted, 0.25)
    assert np.max(np.abs(a - b)) > 0.1
    # the padded keys really are ignored: dropping them gives the same answer
    c, _ = oracle.attn(inp.q, inp.k[:, :, :44], inp.v[:, :, :44], None, 0.25)
    np.testing.assert_allclose(a, c, rtol=1e-13, atol=1e-14)


def test_fully_masked_row_is_zero_with_neg_inf_lse():
    inp = workloads.make_attn(2, 2, 2, 4, 10, 8, dtype=torch.float32, n_pad=[10, 0], seed=6)
    out, lse = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.5)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(out[1])) and np.all(np.isfinite(lse[1]))


def test_empty_key_set():
    q = torch.randn(1, 1, 3, 8)
    k = torch.zeros(1, 1, 0, 8)
    out, lse = oracle.attn(q, k, k, None, 0.5)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# --------------------------------------------------------------------------
# LSE merge
# --------------------------------------------------------------------------
@pytest.mark.parametrize("cuts", [[0, 30, 61], [0, 1, 61], [0, 20, 40, 61], [0, 61]])
def test_merge_of_chunks_equals_unsplit_attention(cuts):
    """Ring-attention page, accuracy section: merging the (out, lse) of two KV
    chunks gives the single call over all keys."""
    inp = workloads.make_attn(2, 4, 2, 13, 61, 32, dtype=torch.bfloat16, n_pad=[0, 11], seed=9)
    full_o, full_l = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.2)
    outs, lses = [], []
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.attn(inp.q, inp.k[:, :, lo:hi], inp.v[:, :, lo:hi], inp.mask[:, lo:hi], 0.2)
        outs.append(o)
        lses.append(l)
    mo, ml = oracle.merge(outs, lses)
    np.testing.assert_allclose(mo, full_o, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ml, full_l, rtol=1e-12, atol=1e-12)


def test_merge_with_fully_masked_chunk():
    """The second chunk holds only padded keys (lse = -inf): it gets weight 0."""
    inp = workloads.make_attn(1, 2, 2, 6, 50, 16, dtype=torch.float32, n_pad=25, seed=10)
    full_o, full_l = oracle.attn(inp.q, inp.k, inp.v, inp.mask, 0.3)
    o1, l1 = oracle.attn(inp.q, inp.k[:, :, :25], inp.v[:, :, :25], inp.mask[:, :25], 0.3)
    o2, l2 = oracle.attn(inp.q, inp.k[:, :, 25:], inp.v[:, :, 25:], inp.mask[:, 25:], 0.3)
    assert np.all(np.isneginf(l2))
    mo, ml = oracle.merge([o1, o2], [l1, l2])
    np.testing.assert_allclose(mo, full_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ml, full_l, rtol=1e-13, atol=1e-13)
    zo, zl = oracle.merge([o2, o2], [l2, l2])
    assert np.all(zo == 0) and np.all(np.isneginf(zl))


def test_merge_closed_form_and_stability():
    """Two partials with equal lse average to their mean with lse + ln 2; a huge
    lse does not overflow (the max is subtracted first)."""
    o1 = np.array([[1.0, 2.0]])
    o2 = np.array([[3.0, -2.0]])
    mo, ml = oracle.merge([o1, o2], [np.array([5.0]), np.array([5.0])])
    np.testing.assert_allclose(mo, [[2.0, 0.0]], atol=1e-15)
    np.testing.assert_allclose(ml, [5.0 + math.log(2.0)], atol=1e-15)
    mo, ml = oracle.merge([o1, o2], [np.array([1000.0]), np.array([1000.0 - math.log(3.0)])])
    np.testing.assert_allclose(mo, [[1.5, 1.0]], atol=1e-12)
    np.testing.assert_allclose(ml, [1000.0 + math.log(4.0 / 3.0)], atol=1e-12)
    # order does not matter
    a = oracle.merge([o1, o2], [np.array([0.3]), np.array([-1.2])])
    b = oracle.merge([o2, o1], [np.array([-1.2]), np.array([0.3])])
    np.testing.assert_allclose(a[0], b[0], atol=1e-15)


# --------------------------------------------------------------------------
# paged cache: gather, append, decode
# --------------------------------------------------------------------------
def test_block_table_example_from_the_page():
    """Logical blocks [0][1][2] -> physical [9][3][17]: token t of the request
    is read from physical block table[t // 16], slot t % 16."""
    g = _golden("block_table_example.json")
    phys = g["physical_blocks"]
    nb, H, bs, D = 20, 2, 16, 4
    cache = torch.arange(nb * H * bs * D, dtype=torch.int32).reshape(nb, H, bs, D)
    bt = torch.tensor([phys], dtype=torch.int32)
    got = oracle.paged_gather(cache.numpy(), bt, [3 * bs])[0]  # [H, 48, D]
    for t in range(3 * bs):
        np.testing.assert_array_equal(got[:, t, :], cache[phys[t // bs], :, t % bs, :].numpy())
    # token 20 sits in logical block 1 -> physical block 3, slot 4
    np.testing.assert_array_equal(got[:, 20, :], cache[3, :, 4, :].numpy())


def test_scatter_then_gather_roundtrip():
    rng = np.random.default_rng(0)
    B, H, D, bs = 3, 2, 8, 16
    lens = [1, 16, 37]
    nblk = [-(-L // bs) for L in lens]
    perm = rng.permutation(sum(nblk) + 2)
    bt = np.full((B, 4), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    cache = np.full((len(perm), H, bs, D), -7, dtype=np.int16)
    contig = [rng.integers(-1000, 1000, size=(H, L, D), dtype=np.int16) for L in lens]
    for b, L in enumerate(lens):
        for t in range(L):
            cache[bt[b, t // bs], :, t % bs, :] = contig[b][:, t, :]
    got = oracle.paged_gather(cache, bt, lens)
    for b in range(B):
        np.testing.assert_array_equal(got[b], contig[b])


def test_kv_append_writes_exactly_one_slot_per_head():
    cfg = workloads.DecodeConfig("d", 4, 8, 2, 16, 16, 0, 40, 3)
    inp = workloads.make_decode_inputs(cfg, seed=1, ctx=[0, 15, 16, 40])
    kc, vc = oracle.kv_append(inp.k_cache, inp.v_cache, inp.block_table, inp.pos,
                              inp.k_new, inp.v_new)
    k0 = inp.k_cache.view(torch.int16).numpy()
    changed = np.argwhere(kc != k0)
    assert changed.shape[0] <= 4 * 2 * 16
    for b in range(4):
        p = int(inp.pos[b])
        blk = int(inp.block_table[b, p // 16])
        np.testing.assert_array_equal(kc[blk, :, p % 16, :], inp.k_new[b].view(torch.int16).numpy())
        np.testing.assert_array_equal(vc[blk, :, p % 16, :], inp.v_new[b].view(torch.int16).numpy())
    # positions 15 and 16 are the last slot of block 0 and the first of block 1
    assert int(inp.block_table[1, 0]) != int(inp.block_table[2, 1])


def _contiguous_kv(inp, kc, vc):
    """Per-sequence contiguous K/V rebuilt by gathering through the table."""
    ks = oracle.paged_gather(kc, inp.block_table, inp.ctx_lens)
    vs = oracle.paged_gather(vc, inp.block_table, inp.ctx_lens)
    to_t = lambda a: torch.from_numpy(a.copy()).view(torch.bfloat16)
    return [to_t(k) for k in ks], [to_t(v) for v in vs]


@pytest.mark.parametrize("ctx", [[0, 1, 15, 16, 17, 100], [511, 512, 513, 1023, 1024, 2000]])
def test_incremental_decode_equals_full_recompute(ctx):
    """nanoVLM page: after appending the new token's K/V, attending with that
    token's query over the cache equals recomputing the last row of full
    attention over the whole sequence (non-causal and causal agree on the last
    row).  Checked against the oracle's contiguous path and library SDPA."""
    cfg = workloads.DecodeConfig("d", len(ctx), 8, 2, 64, 16, 0, 2048, 5)
    inp = workloads.make_decode_inputs(cfg, seed=2, ctx=ctx)
    kc, vc = oracle.kv_append(inp.k_cache, inp.v_cache, inp.block_table, inp.pos,
                              inp.k_new, inp.v_new)
    kt = torch.from_numpy(kc).view(torch.bfloat16)
    vt = torch.from_numpy(vc).view(torch.bfloat16)
    out, lse = oracle.paged_decode(inp.q, kt, vt, inp.block_table, inp.ctx_lens, inp.scale)
    assert np.all(np.isfinite(out))
    ks, vs = _contiguous_kv(inp, kc, vc)
    for b in range(len(ctx)):
        k = ks[b].unsqueeze(0)  # [1, Hkv, L, D]
        v = vs[b].unsqueeze(0)
        q = inp.q[b].unsqueeze(0).unsqueeze(2)  # [1, Hq, 1, D]
        # the appended token is the last row of the contiguous sequence
        np.testing.assert_array_equal(k[0, :, -1].view(torch.int16).numpy(),
                                      inp.k_new[b].view(torch.int16).numpy())
        ro, rl = oracle.attn(q, k, v, None, inp.scale)
        np.testing.assert_allclose(out[b], ro[0, :, 0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], rl[0, :, 0], rtol=1e-12, atol=1e-13)
        so, sl = _sdpa_f64(q, k, v, None, inp.scale)
        np.testing.assert_allclose(out[b], so[0, :, 0], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], sl[0, :, 0], rtol=1e-12, atol=1e-12)


def test_decode_never_reads_unfilled_slots():
    """Unfilled slots hold NaN; the decode over ctx + 1 tokens after the append
    is finite, and the decode that (wrongly) skips the append reads a NaN."""
    cfg = workloads.DecodeConfig("d", 3, 4, 1, 32, 16, 5, 50, 2)
    inp = workloads.make_decode_inputs(cfg, seed=3)
    out, _ = oracle.paged_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.ctx, inp.scale)
    assert np.all(np.isfinite(out))
    out2, _ = oracle.paged_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.ctx_lens, inp.scale)
    assert np.all(np.isnan(out2))


def test_decode_rejects_bad_block_ids():
    cfg = workloads.DecodeConfig("d", 2, 4, 1, 32, 16, 5, 50, 2)
    inp = workloads.make_decode_inputs(cfg, seed=3)
    bt = inp.block_table.clone()
    bt[1, 0] = inp.num_blocks  # one past the end
    with pytest.raises(ValueError):
        oracle.paged_decode(inp.q, inp.k_cache, inp.v_cache, bt, inp.ctx, inp.scale)


# --------------------------------------------------------------------------
# paged (chunked) prefill
# --------------------------------------------------------------------------
def _prefill_case(B=3, Hq=4, Hkv=2, D=16, T=5, start=(0, 13, 30), bs=16, seed=5, causal=True):
    cfg = workloads.PrefillConfig("p", B, Hq, Hkv, D, T, bs, 0, 0, 3, causal)
    inp = workloads.make_prefill_inputs(cfg, seed=seed, start=start)
    kc, vc = oracle.kv_append_chunk(inp.k_cache, inp.v_cache, inp.block_table, inp.start_pos,
                                    inp.k_new, inp.v_new, block_size=bs)
    kt = torch.from_numpy(kc).view(torch.bfloat16)
    vt = torch.from_numpy(vc).view(torch.bfloat16)
    return inp, kc, vc, kt, vt


def test_kv_append_chunk_equals_token_by_token_appends():
    """A chunk append equals T single-token appends at consecutive positions,
    bit for bit, including chunks that cross block boundaries."""
    inp, kc, vc, _, _ = _prefill_case(T=19, start=(0, 13, 30))
    k_ref, v_ref = oracle._bits(inp.k_cache).copy(), oracle._bits(inp.v_cache).copy()
    for i in range(inp.cfg.T):
        k_ref, v_ref = oracle.kv_append(k_ref, v_ref, inp.block_table, inp.start_pos + i,
                                        inp.k_new[:, :, i].contiguous(), inp.v_new[:, :, i].contiguous())
    np.testing.assert_array_equal(kc, k_ref)
    np.testing.assert_array_equal(vc, v_ref)
    # and every slot after the chunk is still the NaN sentinel
    lens = inp.start_pos + inp.cfg.T
    for b in range(inp.cfg.B):
        t = int(lens[b])
        blk = int(inp.block_table[b, t // 16])
        if t % 16:
            assert np.all(np.isnan(torch.from_numpy(kc[blk, :, t % 16]).view(torch.bfloat16).float().numpy()))


def test_causal_prefill_brute_force_60_digits():
    """Each causal query row against 60-digit brute force over the tokens the
    row may see, gathered from the cache by hand (block, slot) = divmod(t, bs)."""
    bs = 4
    inp, kc, vc, kt, vt = _prefill_case(B=2, Hq=4, Hkv=2, D=4, T=3, start=(0, 6), bs=bs, seed=6)
    out, lse = oracle.paged_prefill(inp.q, kt, vt, inp.block_table, inp.start_pos, True, 0.41, block_size=bs)
    for b in range(2):
        for i in range(3):
            n = int(inp.start_pos[b]) + i + 1
            ks = torch.stack([kt[int(inp.block_table[b, t // bs]), :, t % bs] for t in range(n)], dim=1)
            vs = torch.stack([vt[int(inp.block_table[b, t // bs]), :, t % bs] for t in range(n)], dim=1)
            ro, rl = _mp_attention(inp.q[b:b + 1, :, i:i + 1].float(), ks[None].float(), vs[None].float(),
                                   None, 0.41, 2)
            np.testing.assert_allclose(out[b, :, i], ro[0, :, 0], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(lse[b, :, i], rl[0, :, 0], rtol=1e-12, atol=1e-13)


def test_causal_prefill_from_empty_matches_library_causal_sdpa():
    """A whole prompt (nothing cached before it): PyTorch's fp64 SDPA with
    is_causal=True over the contiguous prompt."""
    inp, _, _, kt, vt = _prefill_case(B=2, Hq=8, Hkv=2, D=32, T=45, start=(0, 0), seed=7)
    out, lse = oracle.paged_prefill(inp.q, kt, vt, inp.block_table, inp.start_pos, True, inp.scale)
    q64 = inp.q.to(torch.float64)
    k64 = inp.k_new.to(torch.float64).repeat_interleave(4, dim=1)
    v64 = inp.v_new.to(torch.float64).repeat_interleave(4, dim=1)
    ref = F.scaled_dot_product_attention(q64, k64, v64, is_causal=True, scale=inp.scale)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)
    # closed form: the first prompt token sees only itself
    np.testing.assert_allclose(out[:, :, 0], v64[:, :, 0].numpy(), rtol=0, atol=1e-15)
    s00 = inp.scale * (q64[:, :, 0] * k64[:, :, 0]).sum(-1)
    np.testing.assert_allclose(lse[:, :, 0], s00.numpy(), rtol=1e-14, atol=1e-14)


def test_chunked_prefill_equals_unchunked():
    """"LLM inference memory accounting", chunked prefill: splitting a prompt
    into chunks changes the schedule, not the result.  Prefilling the last T
    tokens after S cached ones equals the last T rows of prefilling all S + T
    at once."""
    S, T = 37, 22
    whole, _, _, kt, vt = _prefill_case(B=1, Hq=4, Hkv=1, D=16, T=S + T, start=(0,), seed=8)
    ow, lw = oracle.paged_prefill(whole.q, kt, vt, whole.block_table, whole.start_pos, True, whole.scale)
    st = torch.tensor([S], dtype=torch.int32)
    oc, lc = oracle.paged_prefill(whole.q[:, :, S:], kt, vt, whole.block_table, st, True, whole.scale)
    np.testing.assert_allclose(oc, ow[:, :, S:], rtol=0, atol=0)
    np.testing.assert_allclose(lc, lw[:, :, S:], rtol=0, atol=0)


def test_prefill_rows_match_decode_and_contiguous_attention():
    """Non-causal: every chunk query equals a decode over start + T tokens
    (the decode oracle is pinned above).  Causal: row i equals contiguous
    attention over the first start + i + 1 tokens; its last row equals the
    non-causal last row."""
    inp, kc, vc, kt, vt = _prefill_case(T=7, start=(0, 13, 30), seed=9)
    on, ln = oracle.paged_prefill(inp.q, kt, vt, inp.block_table, inp.start_pos, False, inp.scale)
    oc, lc = oracle.paged_prefill(inp.q, kt, vt, inp.block_table, inp.start_pos, True, inp.scale)
    total = inp.start_pos + 7
    for i in range(7):
        od, ld = oracle.paged_decode(inp.q[:, :, i].contiguous(), kt, vt, inp.block_table, total, inp.scale)
        np.testing.assert_allclose(on[:, :, i], od, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(ln[:, :, i], ld, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(oc[:, :, -1], on[:, :, -1], rtol=1e-13, atol=1e-14)
    ks = oracle.paged_gather(kc, inp.block_table, total)
    vs = oracle.paged_gather(vc, inp.block_table, total)
    for b in range(3):
        for i in (0, 3, 6):
            n = int(inp.start_pos[b]) + i + 1
            k = torch.from_numpy(ks[b][:, :n].copy()).view(torch.bfloat16)[None]
            v = torch.from_numpy(vs[b][:, :n].copy()).view(torch.bfloat16)[None]
            ro, rl = oracle.attn(inp.q[b:b + 1, :, i:i + 1], k, v, None, inp.scale)
            np.testing.assert_allclose(oc[b, :, i], ro[0, :, 0], rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(lc[b, :, i], rl[0, :, 0], rtol=1e-13, atol=1e-14)
    # nothing after the chunk is ever read: those slots are NaN
    assert np.all(np.isfinite(on)) and np.all(np.isfinite(oc))


# --------------------------------------------------------------------------
# INT8 KV
# --------------------------------------------------------------------------
def _check_q8_pins(quant):
    """The quantiser pins, against any candidate implementation `quant`."""
    g = torch.Generator().manual_seed(13)
    x = torch.randn(6, 4, 128, generator=g).to(torch.bfloat16)
    x[0, 0] = 0.0  # an all-zero row
    q, s = quant(x)
    xf = x.float().numpy()
    assert q.dtype == np.int8 and np.abs(q.astype(np.int32)).max() <= 127
    # the largest |x| of a row maps to +-127 exactly, and the zero row to 0 / 0
    am = np.abs(xf).argmax(-1)
    for i in range(6):
        for h in range(4):
            if i == 0 and h == 0:
                assert s[i, h] == 0 and not q[i, h].any()
                continue
            assert abs(int(q[i, h, am[i, h]])) == 127
            assert np.sign(q[i, h, am[i, h]]) == np.sign(xf[i, h, am[i, h]])
    # every element within half a step of its row's scale (plus the float32
    # rounding of x / scale, < 1e-5 of a step for |x / scale| <= 127)
    err = np.abs(q.astype(np.float64) * s[..., None].astype(np.float64) - xf)
    assert np.all(err <= 0.5 * s[..., None].astype(np.float64) * (1 + 1e-4) + 1e-30)
    # hand-computed: scale 127/127 = 1 and ties round half to even
    t = torch.tensor([[[127.0, 0.5, 1.5, 2.5, -0.5, -3.5, 126.5, 0.0]]])
    qt, st = quant(t)
    assert float(st[0, 0]) == 1.0
    assert qt[0, 0].tolist() == [127, 0, 2, 2, 0, -4, 126, 0]
    # a row twice as large: the same codes and twice the scale (exact in binary)
    q2, s2 = quant(x * 2)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, 2 * s)


def test_q8_quantiser_pins():
    _check_q8_pins(oracle.quantize_rows_q8)


def test_q8_quantiser_matches_library_int8_quantisation():
    """PyTorch's per-tensor qint8 quantiser with the same scale (it multiplies by
    the reciprocal where the oracle divides, so codes may differ by one only
    where x / scale lies within float rounding of a half)."""
    g = torch.Generator().manual_seed(14)
    x = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    q, s = oracle.quantize_rows_q8(x)
    for r in range(64):
        tq = torch.quantize_per_tensor(x[r].float(), float(s[r]), 0, torch.qint8).int_repr().numpy()
        d = np.abs(tq.astype(np.int32) - q[r].astype(np.int32))
        assert d.max() <= 1
        ratio = x[r].float().numpy() / s[r]
        assert np.all(np.abs(np.abs(ratio[d == 1] - np.floor(ratio[d == 1])) - 0.5) < 1e-4)


def test_q8_planted_mistakes_are_caught():
    def per_tensor(x):  # one scale for the whole tensor instead of one per row
        xs = x.float().numpy()
        s = np.float32(np.abs(xs).max() / np.float32(127))
        q = np.clip(np.rint(xs / s), -127, 127).astype(np.int8)
        return q, np.full(xs.shape[:-1], s, dtype=np.float32)
    def scale_128(x):
        xs = x.float().numpy()
        s = (np.abs(xs).max(-1) / np.float32(128)).astype(np.float32)
        q = np.clip(np.rint(xs / np.where(s > 0, s, 1)[..., None]), -127, 127).astype(np.int8)
        return q, s
    def truncate(x):
        xs = x.float().numpy()
        s = (np.abs(xs).max(-1) / np.float32(127)).astype(np.float32)
        q = np.clip(np.trunc(xs / np.where(s > 0, s, 1)[..., None]), -127, 127).astype(np.int8)
        return q, s
    def half_up(x):
        xs = x.float().numpy()
        s = (np.abs(xs).max(-1) / np.float32(127)).astype(np.float32)
        q = np.clip(np.floor(xs / np.where(s > 0, s, 1)[..., None] + 0.5), -127, 127).astype(np.int8)
        return q, s
    for bad in (per_tensor, scale_128, truncate, half_up):
        with pytest.raises(AssertionError):
            _check_q8_pins(bad)


def test_q8_append_writes_one_quantised_row_per_head():
    cfg = workloads.DecodeConfig("q", 5, 8, 2, 64, 16, 0, 100, 3)
    d = workloads.make_decode_inputs_q8(cfg, seed=15, ctx=[0, 15, 16, 17, 100])
    pos = d.pos.clone()
    pos[3] = -1  # idle
    kq, vq, ks, vs = oracle.kv_append_q8(d.kq_cache, d.vq_cache, d.k_scale, d.v_scale, d.block_table, pos,
                                         d.k_new, d.v_new)
    qk, sk = oracle.quantize_rows_q8(d.k_new)
    changed = ((kq != d.kq_cache.numpy()).any(axis=(1, 3)) |
               ~np.isclose(ks, d.k_scale.numpy(), equal_nan=True).all(axis=1))
    for b in range(5):
        if b == 3:
            continue
        blk, slot = int(d.block_table[b, int(pos[b]) // 16]), int(pos[b]) % 16
        np.testing.assert_array_equal(kq[blk, :, slot], qk[b])
        np.testing.assert_array_equal(ks[blk, :, slot], sk[b])
        assert changed[blk, slot]
        changed[blk, slot] = False
    assert not changed.any()  # nothing else, and nothing for the idle sequence


def test_q8_decode_on_exactly_representable_cache_equals_bf16_decode():
    """Rows of integers times 1/4 with one element +-127/4: quantisation is
    exact, so the INT8 decode equals the (pinned) bf16 decode on the same
    values, to the last bit of fp64."""
    cfg = workloads.DecodeConfig("q", 3, 8, 2, 64, 16, 0, 300, 2)
    d = workloads.make_decode_inputs(cfg, seed=16, ctx=[10, 100, 300])
    g = torch.Generator().manual_seed(17)
    def exact_rows(shape):
        v = torch.randint(-126, 127, shape, generator=g).float()
        v[..., 0] = 127.0
        return (v / 4).to(torch.bfloat16)
    kc = exact_rows(d.k_cache.shape)
    vc = exact_rows(d.v_cache.shape)
    kq, ks = oracle.quantize_rows_q8(kc)
    vq, vs = oracle.quantize_rows_q8(vc)
    assert np.all(ks == 127 / 4 / 127) and np.all(vs == 0.25)
    o8, l8 = oracle.paged_decode_q8(d.q, kq, vq, ks, vs, d.block_table, d.ctx, d.scale)
    o, l = oracle.paged_decode(d.q, kc, vc, d.block_table, d.ctx, d.scale)
    np.testing.assert_array_equal(o8, o)
    np.testing.assert_array_equal(l8, l)


# --------------------------------------------------------------------------
# the pages' worked numbers
# --------------------------------------------------------------------------
def test_kv_bytes_per_token_worked_example():
    g = _golden("pages_numbers.json")
    s = oracle.ModelShape(**g["kv_bytes_per_token_gqa"]["shape"])
    assert s.kv_bytes_per_token() == g["kv_bytes_per_token_gqa"]["value"]
    assert s.sequence_kv_bytes(8192) == g["kv_bytes_8k_sequence_gqa"]["value"]
    mha = oracle.ModelShape(**g["kv_bytes_per_token_mha"]["shape"])
    assert mha.kv_bytes_per_token() == g["kv_bytes_per_token_mha"]["value"]
    mqa = oracle.ModelShape(32, 1, 128, 2)
    assert mqa.kv_bytes_per_token() / s.kv_bytes_per_token() == g["kv_bytes_per_token_mqa_ratio"]["value"]
    assert round(32 * s.sequence_kv_bytes(8192) / 2**30) == g["kv_raw_32_sequences_8k_gib"]["value"]
    cap = g["token_capacity_24gib_pool"]
    assert oracle.token_capacity(cap["pool_gib"] * 2**30, cap["kv_kib_per_token"] * 1024) == cap["value"]
    # the decode workload's cache: one layer, 8 KV heads, D 128, bf16
    assert oracle.ModelShape(1, 8, 128, 2).kv_bytes_per_token() == 4096


def test_score_matrix_sizes_from_the_page():
    g = _golden("pages_numbers.json")
    e = g["score_matrix_3mp_bf16_gb"]
    assert round(oracle.score_matrix_bytes(e["heads"], e["P"], e["elem_bytes"]) / 1e9, 2) == e["value"]
    e = g["score_matrix_cpu_p1024_f32_mib"]
    assert oracle.score_matrix_bytes(e["heads"], e["P"], e["elem_bytes"]) == e["value"] * 2**20
    e = g["score_matrix_8mp_bf16_gib"]
    # 30.75 GiB corresponds to P of about 32 thousand (32,122)
    p = math.sqrt(e["value"] * 2**30 / (e["heads"] * e["elem_bytes"]))
    assert 32000 <= p < 32200
    # the large-image workload (P = 32000) would need about 30.5 GiB
    assert abs(oracle.score_matrix_bytes(16, 32000, 2) / 2**30 - 30.52) < 0.01
    # the MultiheadAttention extra VRAM at 3 MP is about four such matrices
    pts = g["mha_extra_vram_points"]
    ratio = pts["gb"][-1] * 1e9 / oracle.score_matrix_bytes(16, pts["P"][-1], 2)
    assert 3.5 < ratio < 4.5


# --------------------------------------------------------------------------
# the pins catch plausible mistakes
# --------------------------------------------------------------------------
def _mutant(tmp_path, find, replace, name):
    """A copy of the oracle library with one planted mistake."""
    import ctypes
    import subprocess
    src = open(oracle._SRC).read()
    assert find in src, find
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(find, replace, 1))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so),
                    str(path), "-lm"], check=True)
    return ctypes.CDLL(str(so))


MUTANTS = [
    ("mask_scaled", "s[j] = scale * dot + (mask ? (double)mask[j] : 0.0);",
     "s[j] = scale * (dot + (mask ? (double)mask[j] : 0.0));"),
    ("mask_dropped", "s[j] = scale * dot + (mask ? (double)mask[j] : 0.0);",
     "s[j] = scale * dot;"),
    ("lse_log2", "*lse = m + log(l);", "*lse = m + log2(l);"),
    ("lse_no_max", "*lse = m + log(l);", "*lse = log(l);"),
    ("gqa_modulo", "int64_t g = h / group;\n            for (int64_t d = 0; d < D; ++d)\n                qv[d]",
     "int64_t g = h % Hkv;\n            for (int64_t d = 0; d < D; ++d)\n                qv[d]"),
    ("value_uses_key", "out[d] += s[j] * widen(v, kv_dtype, val_index[j] + d);",
     "out[d] += s[j] * widen(k, kv_dtype, key_index[j] + d);"),
    ("no_normalise", "for (int64_t d = 0; d < D; ++d) out[d] /= l;", ""),
    ("decode_slot_reversed", "((blk * Hkv + g) * block_size + t % block_size) * D",
     "((blk * Hkv + g) * block_size + (block_size - 1 - t % block_size)) * D"),
    ("decode_head_modulo", "int64_t b = bh / Hq, h = bh % Hq, g = h / group;",
     "int64_t b = bh / Hq, h = bh % Hq, g = h % Hkv;"),
    ("decode_block_index", "int64_t blk = block_table[b * bt_stride + t / block_size];",
     "int64_t blk = block_table[b * bt_stride + t % block_size];"),
    ("prefill_causal_off_by_one", "int64_t n = causal ? start + i + 1 : total;",
     "int64_t n = causal ? start + i : total;"),
    ("prefill_causal_ignores_start", "int64_t n = causal ? start + i + 1 : total;",
     "int64_t n = causal ? i + 1 : total;"),
    ("prefill_noncausal_drops_chunk", "int64_t n = causal ? start + i + 1 : total;",
     "int64_t n = causal ? start + i + 1 : start + 1;"),
    ("prefill_query_row", "qv[d] = widen(q, q_dtype, r * D + d);",
     "qv[d] = widen(q, q_dtype, (r - i) * D + d);"),
]


@pytest.mark.parametrize("name,find,replace", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistakes_are_caught(tmp_path, monkeypatch, name, find, replace):
    lib = _mutant(tmp_path, find, replace, name)
    real = oracle._load()
    lib.oracle_attn.restype = real.oracle_attn.restype
    lib.oracle_attn.argtypes = real.oracle_attn.argtypes
    lib.oracle_paged_decode.restype = real.oracle_paged_decode.restype
    lib.oracle_paged_decode.argtypes = real.oracle_paged_decode.argtypes
    lib.oracle_paged_prefill.restype = real.oracle_paged_prefill.restype
    lib.oracle_paged_prefill.argtypes = real.oracle_paged_prefill.argtypes
    lib.oracle_num_threads.restype = real.oracle_num_threads.restype
    monkeypatch.setattr(oracle, "_lib", lib)
    caught = False
    for check in (lambda: test_attn_brute_force_60_digits(4, 2),
                  lambda: test_attn_matches_library_sdpa(torch.float32, 2, 4, 1, 17, 130, 64, [0, 129]),
                  lambda: test_merge_of_chunks_equals_unsplit_attention([0, 30, 61]),
                  lambda: test_incremental_decode_equals_full_recompute([0, 1, 15, 16, 17, 100]),
                  test_causal_prefill_brute_force_60_digits,
                  test_prefill_rows_match_decode_and_contiguous_attention):
        try:
            check()
        except (AssertionError, ValueError):
            caught = True
            break
    assert caught, f"planted mistake {name} was not caught"
