"""The ring-attention schedule (masked_attention_paged_gb300.ring) on CPU
gloo ranks, as "[sglang] ROCm aiter ring attention" (sections 1-2) lays it
out: each rank attends its own query chunk over every rank's K/V chunk as the
chunks travel once around the ring, merging partials through their LSE.  The
per-chunk attention and the merge are the oracle's here (the library's
kernels need a GPU, and these runs have one GPU per box); the test checks the
exchange, the order the chunks arrive in and the merged result against
attention over the whole sequence."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, T, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    import workloads
    from masked_attention_paged_gb300.ring import RingStaging, ring_attn
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, Hkv, D = 4, 2, 16
    full = workloads.make_attn(1, H, Hkv, world * T, world * T, D, dtype=torch.float32, with_mask=False, seed=61)
    sl = slice(rank * T, (rank + 1) * T)
    q, k, v = full.q[:, :, sl], full.k[:, :, sl], full.v[:, :, sl]
    seen = []

    def attn_fn(q_, k_, v_, scale, bufs):
        # which rank's chunk is this?  (each chunk's first key row identifies it)
        src = [s for s in range(world) if torch.equal(k_[0, 0, 0], full.k[0, 0, s * T])]
        seen.append(src[0] if len(src) == 1 else -1)
        o, l = oracle.attn(q_, k_, v_, None, scale)
        return torch.from_numpy(o), torch.from_numpy(l)

    def merge_fn(outs, lses, bufs):
        o, l = oracle.merge([x.numpy() for x in outs], [x.numpy() for x in lses])
        return torch.from_numpy(o), torch.from_numpy(l)

    staging = RingStaging(q, k)
    o, l = ring_attn(q, k, v, full.scale, staging=staging, attn_fn=attn_fn, merge_fn=merge_fn)
    ro, rl = oracle.attn(q, full.k, full.v, None, full.scale)
    out[rank] = (float(np.abs(o.numpy() - ro).max()), float(np.abs(l.numpy() - rl).max()), seen)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_attention_schedule_on_gloo_ranks(world):
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, 37, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    for r in range(world):
        err_o, err_l, seen = out[r]
        assert err_o < 1e-12 and err_l < 1e-12, (r, err_o, err_l)
        # the chunks arrive from rank r, r - 1, r - 2, ... (mod world), each once
        assert seen == [(r - s) % world for s in range(world)], (r, seen)
