"""GPU parity of masked attention (attn_fwd) and the LSE merge against the
oracle: every output element at sizes spanning several 128-row/128-key
tiles with ragged tails, and sampled rows at the full workloads (patch
attention P = 1944 and P = 32000, packed T = 32760 chunked attention merged
through the LSE)."""
import math

import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(inp, out_dtype=None, bounds=False):
    """attn_fwd on the GPU; bounds=True gives it the workspace with room for
    the per-tile key bounds (the D = 64 kernel then skips its max pass where
    they rule out overflow), False the bare status word."""
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    mask = inp.mask.to(DEV) if inp.mask is not None else None
    out = None
    if out_dtype is not None:
        out = torch.empty(q.shape, dtype=out_dtype, device=DEV)
    B, Hkv, Pk, D = k.shape
    ws = lib.Workspace(lib.attn_fwd_workspace_size_for(B, Hkv, Pk, D) if bounds else 256)
    o, l = lib.attn_fwd(q, k, v, mask, inp.scale, out=out, workspace=ws)
    assert ws.status() == 0
    return o, l


def test_tiny_f32_workload_full():
    """fp32 inputs, B1 H16 P512 D64, last 37 keys padded: every element within 1e-4."""
    inp = workloads.make_attn_inputs(workloads.ATTN_CONFIGS["tiny_f32"], seed=0)
    o, l = _run(inp)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro, fp32_inputs=True)
    assert_lse_close(l, rl)


@pytest.mark.parametrize("B,Hq,Hkv,Pq,Pk,D,pad", [
    (1, 2, 2, 1, 1, 32, 0),
    (2, 4, 2, 77, 130, 64, [0, 129]),
    (1, 3, 1, 129, 257, 96, 5),
    (1, 2, 2, 200, 64, 128, 63),
])
def test_f32_small_shapes(B, Hq, Hkv, Pq, Pk, D, pad):
    inp = workloads.make_attn(B, Hq, Hkv, Pq, Pk, D, dtype=torch.float32, n_pad=pad, seed=1)
    o, l = _run(inp)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro, fp32_inputs=True)
    assert_lse_close(l, rl)


@pytest.mark.parametrize("B,Hq,Hkv,Pq,Pk,D,pad", [
    (1, 1, 1, 128, 128, 64, 0),         # exactly one tile
    (1, 2, 2, 1, 1, 64, 0),             # a single query and key
    (1, 2, 1, 127, 129, 64, 0),         # ragged on both sides, GQA
    (2, 4, 2, 300, 555, 64, [37, 0]),   # several tiles, per-batch padding
    (1, 4, 4, 129, 1000, 128, 100),     # D 128
    (1, 2, 2, 513, 257, 128, [0]),      # Pq > Pk
    (3, 2, 1, 64, 700, 128, [1, 128, 300]),
])
@pytest.mark.parametrize("bounds", [False, True])
def test_bf16_tensor_core_small_shapes(B, Hq, Hkv, Pq, Pk, D, pad, bounds):
    inp = workloads.make_attn(B, Hq, Hkv, Pq, Pk, D, dtype=torch.bfloat16, n_pad=pad, seed=2)
    o, l = _run(inp, bounds=bounds)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro)
    assert_lse_close(l, rl)


def test_bf16_no_mask_f32_output_and_finite_mask_values():
    inp = workloads.make_attn(1, 2, 2, 150, 300, 64, dtype=torch.bfloat16, seed=3, with_mask=False)
    o, l = _run(inp, out_dtype=torch.float32)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, None, inp.scale)
    assert_out_close(o, ro)
    assert_lse_close(l, rl)
    inp.mask = torch.randn(1, 300) * 2.0  # arbitrary finite additive values
    inp.mask[0, 250:] = float("-inf")
    o, l = _run(inp)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro)
    assert_lse_close(l, rl)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fully_masked_rows_and_empty_keys(dtype):
    inp = workloads.make_attn(2, 2, 2, 70, 200, 64, dtype=dtype, n_pad=[200, 10], seed=4)
    o, l = _run(inp)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(l[0]))
    ro, rl = oracle.attn(inp.q[1:], inp.k[1:], inp.v[1:], inp.mask[1:], inp.scale)
    assert_out_close(o[1:], ro, fp32_inputs=dtype == torch.float32)
    assert_lse_close(l[1:], rl)
    q = inp.q.to(DEV)
    k0 = torch.empty(2, 2, 0, 64, dtype=dtype, device=DEV)
    o, l = lib.attn_fwd(q, k0, k0, None, 0.125)
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))


@pytest.mark.parametrize("bounds", [False, True])
@pytest.mark.parametrize("D,gain", [(64, 40.0), (128, 40.0), (64, 6.0), (128, 6.0), (64, 2.5)])
def test_score_jump_after_the_first_tile(D, gain, bounds):
    """Keys of later tiles scaled up so their scores exceed the first tile's
    by tens (gain 6) to hundreds (gain 40) of log2 units: the kernel's
    exponentials against the running reference overflow (to beyond 2^64, or
    to +inf), and its fallback (S reloaded, or recomputed from Q and K in
    shared memory when S's columns are already reused) must still give the
    softmax of the definition."""
    inp = workloads.make_attn(2, 4, 2, 300, 700, D, dtype=torch.bfloat16, n_pad=[0, 37], seed=41)
    k = inp.k.float()
    k[:, :, 128:384] *= gain  # tiles 1 and 2
    k[:, 1, 600:] *= gain  # and a late tile of one head
    inp.k = k.to(torch.bfloat16)
    o, l = _run(inp, bounds=bounds)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    g = o.float().cpu().numpy()
    assert np.all(np.isfinite(g))
    # Such peaked rows return nearly one V row, up to |v| ~ 4.7, where bf16's
    # own rounding of the output (half an ulp, 2^-9 relative) plus that of P
    # (2^-9 of |v|) can pass 2e-2 on their own: the bound grows with |ref|
    # by 2^-8, which a wrong fallback (wrong weights, O(1) errors) still fails.
    err = np.abs(g - ro)
    assert np.all(err <= 2e-2 + np.abs(ro) / 256), f"jump D={D} gain={gain}: max abs err {err.max():.3g}"
    assert err.mean() <= 2e-3 + np.abs(ro).mean() / 256
    assert_lse_close(l, rl, what=f"jump lse D={D} gain={gain}")


@pytest.mark.parametrize("gain", [1.0, 3.0, 8.0])
def test_key_bound_path_at_its_threshold(gain):
    """D = 64 at the size where attn_fwd starts using the per-tile key bounds
    (B Hq Pq Pk D = 2^36): the bound-certified tiles skip the max pass, the
    rest (later tiles' keys scaled by `gain`, and the padded tail) take the
    full path; sampled rows of every head against the oracle."""
    inp = workloads.make_attn(1, 16, 8, 8192, 8192, 64, dtype=torch.bfloat16, n_pad=300, seed=43)
    k = inp.k.float()
    k[:, :, 4096:] *= gain
    inp.k = k.to(torch.bfloat16)
    o, l = _run(inp, bounds=True)
    rows = sample_rows(1, 16, 8192, 256, seed=12)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale, rows=rows)
    g = o.reshape(-1, 64)[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
    assert_lse_close(l.reshape(-1)[torch.from_numpy(rows).to(DEV)], rl)
    if gain == 1.0:
        # ordinary N(0, 1) inputs: the bf16 bars as stated
        assert_out_close(g, ro, what="key-bound path, gain 1")
        return
    # later tiles scaled up: peaked rows, where the bound grows with |ref|
    # (see test_score_jump_after_the_first_tile)
    err = np.abs(g - ro)
    assert np.all(np.isfinite(g))
    assert np.all(err <= 2e-2 + np.abs(ro) / 256), f"gain {gain}: max abs err {err.max():.3g}"
    assert err.mean() <= 2e-3 + np.abs(ro).mean() / 256


@pytest.mark.parametrize("D", [64, 128])
def test_last_wave_split_over_key_tiles(D):
    """160 query-tile pairs on a GPU of fewer SMs: the units of the last,
    partial wave are each split over their key tiles and merged through the
    LSE; every output element against the oracle (ragged keys, padding and
    GQA included)."""
    inp = workloads.make_attn(1, 160, 32, 200, 1000, D, dtype=torch.bfloat16, n_pad=77, seed=44)
    o, l = _run(inp, bounds=True)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro, what=f"split D={D}")
    assert_lse_close(l, rl, what=f"split lse D={D}")
    # and the same through the bare status-word workspace (no split)
    o2, l2 = _run(inp, bounds=False)
    assert (o2.float() - o.float()).abs().max().item() <= 2e-2
    assert (l2 - l).abs().max().item() <= 1e-3


def test_patch_small_workload_full():
    """B1 H16 P1944 D64 bf16 with a seeded 0-64 padded tail: every element."""
    inp = workloads.make_attn_inputs(workloads.ATTN_CONFIGS["patch_small"], seed=0)
    o, l = _run(inp, bounds=True)  # the workspace bench.py gives it
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(o, ro)
    assert_lse_close(l, rl)


def test_patch_large_workload_sampled():
    """B1 H16 P32000 D64 bf16, last 128 keys padded: 2048 seeded query rows
    (the split last wave's rows among them)."""
    inp = workloads.make_attn_inputs(workloads.ATTN_CONFIGS["patch_large"], seed=0)
    o, l = _run(inp, bounds=True)  # the workspace bench.py gives it
    rows = sample_rows(1, 16, 32000, 2048, seed=11)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale, rows=rows)
    assert_out_close(o.reshape(-1, 64)[torch.from_numpy(rows).to(DEV)], ro)
    assert_lse_close(l.reshape(-1)[torch.from_numpy(rows).to(DEV)], rl)


@pytest.mark.parametrize("dtype,n", [(torch.bfloat16, 2), (torch.float32, 2), (torch.float32, 3), (torch.bfloat16, 4),
                                     (torch.bfloat16, 5)])
def test_lse_merge_against_oracle(dtype, n):
    """Chunk partials from the oracle, merged on the GPU, against the oracle's
    merge; one chunk holds only padded keys so its lse is -inf."""
    inp = workloads.make_attn(2, 4, 4, 90, 50 * n, 128, dtype=torch.float32, n_pad=[0, 50], seed=5)
    outs, lses = [], []
    for c in range(n):
        sl = slice(50 * c, 50 * (c + 1))
        o, l = oracle.attn(inp.q, inp.k[:, :, sl], inp.v[:, :, sl], inp.mask[:, sl], inp.scale)
        outs.append(o)
        lses.append(l)
    g_outs = [torch.from_numpy(o).to(dtype).to(DEV) for o in outs]
    g_lses = [torch.from_numpy(l).float().contiguous().to(DEV) for l in lses]
    mo, ml = lib.attn_lse_merge(g_outs, g_lses)
    # the oracle merges exactly the values the GPU was given
    ro, rl = oracle.merge([t.float().cpu().numpy() for t in g_outs], [t.cpu().numpy() for t in g_lses])
    assert_out_close(mo, ro, fp32_inputs=dtype == torch.float32)
    assert_lse_close(ml, rl)
    full_o, full_l = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(mo, full_o, fp32_inputs=False)
    assert_lse_close(ml, full_l)


@pytest.mark.parametrize("D,n", [(40, 3), (8, 2), (24, 8)])
def test_lse_merge_narrow_heads(D, n):
    """Head dims that are not a multiple of 16 take the 8-elements-per-thread
    form of the merge: seeded partials (one row fully masked in the first)
    against the oracle's merge, P with a ragged tail."""
    g = torch.Generator().manual_seed(60 + D)
    outs = [torch.randn(2, 3, 77, D, generator=g).to(torch.bfloat16) for _ in range(n)]
    lses = [(torch.randn(2, 3, 77, generator=g) * 3).float() for _ in range(n)]
    lses[0][0, 0, 5] = float("-inf")
    mo, ml = lib.attn_lse_merge([o.to(DEV) for o in outs], [l.to(DEV) for l in lses])
    ro, rl = oracle.merge([o.float().numpy() for o in outs], [l.numpy() for l in lses])
    assert_out_close(mo, ro)
    assert_lse_close(ml, rl)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_lse_merge_extreme_lse_spread(dtype):
    """Partials whose LSEs differ by hundreds to a thousand (far past where
    exp of either would overflow or underflow on its own), mixed with -inf
    partials: the merge subtracts the row maximum first, so the result is the
    dominant partial wherever one dominates and a finite mix elsewhere."""
    g = torch.Generator().manual_seed(88)
    n, D = 4, 128
    outs = [torch.randn(1, 3, 150, D, generator=g).to(dtype) for _ in range(n)]
    base = torch.randn(1, 3, 150, generator=g) * 2
    offs = [0.0, -700.0, 350.0, 1000.0]
    lses = [(base + off + torch.randn(1, 3, 150, generator=g)).float() for off in offs]
    lses[3][0, 0, :50] = float("-inf")   # the largest partial absent on some rows
    lses[2][0, 1, ::3] = float("-inf")
    lses[1][0, 2, :] = 1000.0 + base[0, 2]  # a tie with partial 3 on one head
    lses[3][0, 2, :] = 1000.0 + base[0, 2]
    mo, ml = lib.attn_lse_merge([o.to(DEV) for o in outs], [l.to(DEV) for l in lses])
    ro, rl = oracle.merge([o.float().numpy() for o in outs], [l.numpy() for l in lses])
    assert_out_close(mo, ro, fp32_inputs=dtype == torch.float32, what="extreme spread")
    assert_lse_close(ml, rl)


def test_lse_merge_all_partials_masked():
    o = torch.randn(1, 2, 10, 64, device=DEV).to(torch.bfloat16)
    l = torch.full((1, 2, 10), float("-inf"), device=DEV)
    mo, ml = lib.attn_lse_merge([o, o], [l, l.clone()])
    assert torch.all(mo == 0) and torch.all(torch.isneginf(ml))


def test_chunked_packed_workload_sampled():
    """Packed [T=32760, H=24, D=128] bf16, two KV chunks of 16380 keys each
    attended with their LSE, merged on the GPU, against the oracle over all
    keys at 2048 seeded rows (the split last wave's among them); the merge
    also matches the unsplit GPU call."""
    cfg = workloads.ATTN_CONFIGS["chunked"]
    inp = workloads.make_attn_inputs(cfg, seed=0)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)  # [1, H, T, D] views of [T, H, D]
    assert not q.is_contiguous()
    outs, lses = [], []
    for lo, hi in cfg.chunk_bounds():
        o, l = lib.attn_fwd(q, k[:, :, lo:hi], v[:, :, lo:hi], None, inp.scale)
        outs.append(o)
        lses.append(l)
    # packed output buffer [T, H, D] viewed as [1, H, T, D]
    out_packed = torch.empty(cfg.Pq, cfg.Hq, cfg.D, dtype=torch.bfloat16, device=DEV)
    mo, ml = lib.attn_lse_merge(outs, lses, out=out_packed.permute(1, 0, 2).unsqueeze(0))
    rows = sample_rows(1, 24, 32760, 2048, seed=12)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, None, inp.scale, rows=rows)
    ridx = torch.from_numpy(rows).to(DEV)
    assert_out_close(mo.reshape(-1, 128)[ridx] if mo.is_contiguous() else
                     mo.contiguous().reshape(-1, 128)[ridx], ro)
    assert_lse_close(ml.reshape(-1)[ridx], rl)
    full_o, full_l = lib.attn_fwd(q, k, v, None, inp.scale)
    d = (full_o.float() - mo.float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3
    assert (full_l - ml).abs().max().item() <= 1e-3


def test_no_score_matrix_is_allocated():
    """Peak extra device memory of one call is the output and LSE: linear in P.
    The library allocates nothing; a P x P score matrix would dwarf this."""
    extra = {}
    for P in (1944, 3952, 7776, 11616, 16000, 32000):
        inp = workloads.make_attn(1, 16, 16, P, P, 64, dtype=torch.bfloat16, n_pad=13, seed=6)
        q, k, v, m = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.mask.to(DEV)
        ws = lib.Workspace(256)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        free0 = torch.cuda.mem_get_info()[0]
        o, l = lib.attn_fwd(q, k, v, m, inp.scale, workspace=ws)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        extra[P] = torch.cuda.max_memory_allocated() - base
        out_bytes = o.numel() * 2 + l.numel() * 4
        assert extra[P] <= out_bytes + (2 << 20), (P, extra[P], out_bytes)
        # a single bf16 score matrix H x P x P would be 30x (P=1944) to 480x (P=32000)
        # larger than out + lse (the allocator's block rounding can add ~1 MB to the peak)
        assert extra[P] * 20 < oracle.score_matrix_bytes(16, P, 2)
        # nothing outside torch's allocator either (allow allocator granularity)
        assert free0 - free1 <= out_bytes + (64 << 20)
        del o, l
    Ps = np.array(sorted(extra), dtype=float)
    ys = np.array([extra[int(p)] for p in Ps], dtype=float)
    quad = np.polyfit(Ps, ys, 2)[0]
    # one bf16 score matrix of 16 heads is 32 B per P^2; the fit (whose noise is the
    # allocator's 2 MB rounding, about 0.002 B/P^2 over these sizes) must stay under 1% of that
    assert abs(quad) < 0.01 * 16 * 2, quad
