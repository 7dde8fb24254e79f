"""GPU parity of attn_fwd at head_dim 128 without a mask, which runs on CTA
pairs (two SMs' tensor cores multiplying as one, M = 256; each CTA holds one
128-row query tile and half of every K/V tile): every output element and LSE
against the oracle over ragged query and key counts -- query tiles past the
rows, key halves past the keys, score buffers reused across tiles -- GQA,
f32 output, the split last wave, and score jumps that force the full softmax
path and the rescale of O."""
import numpy as np
import pytest
import torch

import masked_attention_paged_gb300 as lib
import oracle
import workloads
from _parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(inp, out_dtype=torch.bfloat16, room=False):
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    out = torch.empty(q.shape, dtype=out_dtype, device=DEV)
    B, Hkv, Pk, D = k.shape
    ws = lib.Workspace(lib.attn_fwd_workspace_size_for(B, Hkv, Pk, D) if room else 256)
    o, l = lib.attn_fwd(q, k, v, None, inp.scale, out=out, workspace=ws)
    assert ws.status() == 0
    return o, l


def _kernels_of(fn):
    """Names of the CUDA kernels fn launches (the profiler's first session in
    a process may record nothing, so it is run twice)."""
    from torch.profiler import ProfilerActivity, profile
    names = []
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fn()
            torch.cuda.synchronize()
        names = [e.key for e in prof.key_averages()]
    return names


@pytest.mark.parametrize("B,Hq,Hkv,Pq,Pk", [
    (1, 2, 2, 256, 128),      # one pair, one key tile
    (1, 2, 1, 300, 1000),     # ragged rows and keys (last tile 104 keys), GQA 2
    (2, 4, 2, 129, 50),       # fewer keys than CTA 0's half: CTA 1's K half is all fill
    (1, 3, 3, 64, 700),       # CTA 1's query tile wholly past the rows
    (3, 8, 2, 513, 257),      # GQA 4, three batches, one key in the last tile
    (1, 2, 2, 1, 1),          # one query, one key
    (1, 2, 2, 640, 384),      # exactly three key tiles: each score buffer once
    (1, 2, 2, 256, 769),      # seven tiles: buffers and the K/V ring reused
    (1, 1, 1, 2000, 4096),    # long rows of keys
])
def test_pair_small_shapes(B, Hq, Hkv, Pq, Pk):
    inp = workloads.make_attn(B, Hq, Hkv, Pq, Pk, 128, dtype=torch.bfloat16, seed=71, with_mask=False)
    o, l = _run(inp)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, None, inp.scale)
    assert_out_close(o, ro, what=f"pair {B},{Hq},{Hkv},{Pq},{Pk}")
    assert_lse_close(l, rl, what=f"pair lse {B},{Hq},{Hkv},{Pq},{Pk}")


def test_pair_kernel_is_what_runs():
    """The unmasked D = 128 call launches the CTA-pair kernel; a masked one
    the one-CTA kernel."""
    inp = workloads.make_attn(1, 4, 4, 300, 500, 128, dtype=torch.bfloat16, seed=72)
    q, k, v, m = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.mask.to(DEV)
    names = _kernels_of(lambda: lib.attn_fwd(q, k, v, None, inp.scale))
    assert any("attn_fwd_pair_kernel" in n for n in names), names
    names = _kernels_of(lambda: lib.attn_fwd(q, k, v, m, inp.scale))
    assert any("attn_fwd_tc_kernel" in n for n in names) and not any("pair" in n for n in names), names


def test_pair_f32_output_and_packed_layout():
    """f32 output; q, k, v as [1, H, T, D] views of packed [T, H, D] tensors."""
    inp = workloads.make_attn(1, 6, 3, 450, 333, 128, dtype=torch.bfloat16, seed=73, with_mask=False)
    o, l = _run(inp, out_dtype=torch.float32)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, None, inp.scale)
    assert_out_close(o, ro, what="pair f32 out")
    assert_lse_close(l, rl)
    pq, pk, pv = (t[0].permute(1, 0, 2).contiguous().to(DEV) for t in (inp.q, inp.k, inp.v))
    q, k, v = (t.permute(1, 0, 2).unsqueeze(0) for t in (pq, pk, pv))
    assert not q.is_contiguous()
    o2, l2 = lib.attn_fwd(q, k, v, None, inp.scale)
    assert_out_close(o2, ro, what="pair packed")
    assert_lse_close(l2, rl)


def test_pair_last_wave_split():
    """160 units (query-row pairs of tiles x heads) on a GPU that holds fewer
    clusters: the last wave's units split over their key tiles and merged;
    every element against the oracle, and against the call without room for
    the split."""
    inp = workloads.make_attn(1, 160, 32, 200, 1000, 128, dtype=torch.bfloat16, seed=74, with_mask=False)
    o, l = _run(inp, room=True)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, None, inp.scale)
    assert_out_close(o, ro, what="pair split")
    assert_lse_close(l, rl, what="pair split lse")
    o2, l2 = _run(inp, room=False)
    assert (o2.float() - o.float()).abs().max().item() <= 2e-2
    assert (l2 - l).abs().max().item() <= 1e-3


@pytest.mark.parametrize("gain", [6.0, 40.0])
def test_pair_score_jump(gain):
    """Later key tiles scaled so their scores exceed the running reference by
    tens to hundreds of log2 units: the optimistic tiles fail their row-sum
    check, the full path moves the reference and O is rescaled in TMEM while
    the next tiles' scores already sit in the other buffers."""
    inp = workloads.make_attn(2, 4, 2, 300, 900, 128, dtype=torch.bfloat16, seed=75, with_mask=False)
    k = inp.k.float()
    k[:, :, 128:384] *= gain
    k[:, 1, 700:] *= gain
    inp.k = k.to(torch.bfloat16)
    o, l = _run(inp)
    ro, rl = oracle.attn(inp.q, inp.k, inp.v, None, inp.scale)
    g = o.float().cpu().numpy()
    assert np.all(np.isfinite(g))
    # peaked rows return nearly one V row: the bound grows with |ref| by 2^-8
    # (bf16 rounding of the output and of P), as for the one-CTA kernel
    err = np.abs(g - ro)
    assert np.all(err <= 2e-2 + np.abs(ro) / 256), f"pair jump gain={gain}: max abs err {err.max():.3g}"
    assert err.mean() <= 2e-3 + np.abs(ro).mean() / 256
    assert_lse_close(l, rl, what=f"pair jump lse gain={gain}")


def test_pair_matches_the_one_cta_kernel_with_a_zero_mask():
    """An all-zero additive mask sends the same call to the one-CTA kernel:
    the two kernels agree within the bf16 bars."""
    inp = workloads.make_attn(1, 8, 2, 1000, 1500, 128, dtype=torch.bfloat16, seed=76, with_mask=False)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    o1, l1 = lib.attn_fwd(q, k, v, None, inp.scale)
    zero = torch.zeros(1, 1500, dtype=torch.float32, device=DEV)
    o2, l2 = lib.attn_fwd(q, k, v, zero, inp.scale)
    d = (o1.float() - o2.float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3
    assert (l1 - l2).abs().max().item() <= 1e-3
