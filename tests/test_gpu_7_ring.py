"""Ring attention (masked_attention_paged_gb300.ring) on the library's own
kernels: "[sglang] ROCm aiter ring attention and K/V buffer reuse", sections
1-2.  Two and three gloo ranks share one GPU for the compute while the K/V
chunks travel between them through pinned host buffers; each hop's chunk is
attended with attn_fwd (float32 partials with their LSE), folded into a
float32 running result with attn_lse_merge, and the last merge rounds into
the bf16 output.  The ranks' kernels never wait on one another: every
exchange is a host-side gloo transfer.  Each rank's output and LSE are
compared with the oracle's attention of its queries over the whole sequence;
a direct test of the merge with float32 partials and a bf16 output sits
beside it."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, T, D, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    import torch.distributed as dist

    import masked_attention_paged_gb300 as lib
    import oracle
    import workloads
    from masked_attention_paged_gb300.ring import RingStaging, ring_attn
    torch.cuda.set_device(0)
    lib.load()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, Hkv = 4, 2
    full = workloads.make_attn(1, H, Hkv, world * T, world * T, D, dtype=torch.bfloat16, with_mask=False,
                               seed=70 + world)
    sl = slice(rank * T, (rank + 1) * T)
    q, k, v = (x[:, :, sl].to("cuda") for x in (full.q, full.k, full.v))
    staging = RingStaging(q, k, host=True)
    res = []
    for _ in range(2):  # the staging buffers are reused by the second call
        o, l = ring_attn(q, k, v, full.scale, staging=staging)
        torch.cuda.synchronize()
        res.append((o.float().cpu().numpy(), l.cpu().numpy(), str(o.dtype)))
    ro, rl = oracle.attn(full.q[:, :, sl], full.k, full.v, None, full.scale)
    errs = []
    for o, l, dt in res:
        e = np.abs(o - ro)
        errs.append((float(e.max()), float(e.mean()), float(np.abs(l - rl).max()), bool(np.all(np.isfinite(o))), dt))
    out[rank] = errs
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,T,D", [(2, 300, 128), (3, 257, 64)])
def test_ring_attention_on_the_library_kernels(world, T, D):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, T, D, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    for r in range(world):
        for max_err, mean_err, lse_err, finite, dt in out[r]:
            assert dt == "torch.bfloat16" and finite
            assert max_err <= 2e-2 and mean_err <= 2e-3, (r, max_err, mean_err)
            assert lse_err <= 1e-3, (r, lse_err)


def test_lse_merge_float32_partials_into_bf16_output():
    """float32 partials (as the ring keeps them), merged into a bf16 output:
    the oracle's merge of the same float32 values, and unsplit attention."""
    import masked_attention_paged_gb300 as lib
    import oracle
    import workloads
    from _parity import assert_lse_close, assert_out_close
    inp = workloads.make_attn(2, 3, 3, 133, 3 * 70, 128, dtype=torch.float32, n_pad=[0, 70], seed=71)
    outs, lses = [], []
    for c in range(3):
        sl = slice(70 * c, 70 * (c + 1))
        o, l = oracle.attn(inp.q, inp.k[:, :, sl], inp.v[:, :, sl], inp.mask[:, sl], inp.scale)
        outs.append(torch.from_numpy(o).float().to("cuda"))
        lses.append(torch.from_numpy(l).float().contiguous().to("cuda"))
    mo = torch.empty(outs[0].shape, dtype=torch.bfloat16, device="cuda")
    mo, ml = lib.attn_lse_merge(outs, lses, out=mo)
    assert mo.dtype == torch.bfloat16
    ro, rl = oracle.merge([t.cpu().numpy() for t in outs], [t.cpu().numpy() for t in lses])
    assert_out_close(mo, ro, what="f32 -> bf16 merge")
    assert_lse_close(ml, rl)
    full_o, full_l = oracle.attn(inp.q, inp.k, inp.v, inp.mask, inp.scale)
    assert_out_close(mo, full_o, what="f32 -> bf16 merge vs unsplit")
    assert_lse_close(ml, full_l)
