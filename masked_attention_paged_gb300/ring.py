"""Ring attention over a process group: the sequence-parallel form of
"[sglang] ROCm aiter ring attention and K/V buffer reuse" (sections 1-2).

Each rank holds one contiguous chunk of the sequence: its queries q and its
keys and values k, v.  The K/V chunks travel once around the ring; at every
step a rank attends its own queries over the chunk it holds (attn_fwd, which
returns the chunk's LSE), passes that chunk on to the next rank while it
computes, and folds the chunk's (out, LSE) into its running result with the
LSE merge (attn_lse_merge: out = sum_i exp(lse_i - lse) out_i).  After
world_size steps every rank holds exact non-causal attention of its queries
over the whole sequence.  There is no output exchange.

The K/V chunk in flight lives in a fixed, stacked, double-buffered staging
buffer (RingStaging) that the caller allocates once and reuses on every call,
as the page's K/V buffer reuse does, so a step allocates nothing.  Partial
results and the running merge are kept in float32 and rounded once, by the
last merge, into the output's dtype.

A backend that moves only host memory (gloo) gets the staging buffer in
pinned host memory: each step copies the chunk it holds to one device buffer
for the attention while the host buffers travel, and a host buffer is
received into only once its copy to the device has completed.

attn_fn and merge_fn default to this library's kernels; passing other
functions with the same contract (they return (out, lse)) lets the ring's
schedule be exercised on ranks without a GPU.
"""
from __future__ import annotations

import math
from typing import Callable, Optional, Sequence, Tuple

import torch

Pair = Tuple[torch.Tensor, torch.Tensor]


class RingStaging:
    """Caller-owned buffers of ring_attn, reused on every call: the stacked
    K/V chunk, double-buffered ([2 slots][K, V][...k.shape]), two partial
    (out, lse) pairs and two running-merge pairs in float32.

    host=True keeps the travelling chunk in pinned host memory (for a backend
    that moves only host tensors) plus one device copy of it for the
    attention."""

    def __init__(self, q: torch.Tensor, k: torch.Tensor, host: bool = False):
        dev = q.device
        self.host = bool(host)
        if self.host:
            self.kv = torch.empty((2, 2) + tuple(k.shape), dtype=k.dtype).pin_memory()
            self.kv_dev = torch.empty((2,) + tuple(k.shape), dtype=k.dtype, device=dev)
            self.copied = [None, None]  # event: slot's last device copy has completed
        else:
            self.kv = torch.empty((2, 2) + tuple(k.shape), dtype=k.dtype, device=dev)
            self.kv_dev = None
        self.parts = [(torch.empty(q.shape, dtype=torch.float32, device=dev),
                       torch.empty(q.shape[:3], dtype=torch.float32, device=dev)) for _ in range(2)]
        self.accs = [(torch.empty(q.shape, dtype=torch.float32, device=dev),
                      torch.empty(q.shape[:3], dtype=torch.float32, device=dev)) for _ in range(2)]

    def fits(self, q: torch.Tensor, k: torch.Tensor, host: bool = False) -> bool:
        kv_dev = self.kv_dev.device if self.host else self.kv.device
        return (tuple(self.kv.shape[2:]) == tuple(k.shape) and self.kv.dtype == k.dtype and self.host == host
                and tuple(self.parts[0][0].shape) == tuple(q.shape) and kv_dev == q.device)


def _host_exchange(q: torch.Tensor, group) -> bool:
    """True when the group's backend moves only host tensors and q is on a GPU."""
    import torch.distributed as dist
    return q.is_cuda and dist.get_backend(group) == "gloo"


def _lib_attn(q, k, v, scale, bufs: Pair) -> Pair:
    from . import attn_fwd
    return attn_fwd(q, k, v, None, scale, out=bufs[0], lse=bufs[1])


def _lib_merge(outs: Sequence[torch.Tensor], lses: Sequence[torch.Tensor], bufs: Pair) -> Pair:
    from . import attn_lse_merge
    return attn_lse_merge(outs, lses, out=bufs[0], lse=bufs[1])


def ring_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: Optional[float] = None,
              group=None, staging: Optional[RingStaging] = None, out: Optional[torch.Tensor] = None,
              lse: Optional[torch.Tensor] = None,
              attn_fn: Optional[Callable[..., Pair]] = None,
              merge_fn: Optional[Callable[..., Pair]] = None) -> Pair:
    """Attention of this rank's queries over every rank's keys (non-causal).

    q: [1, H, T_local, D]; k, v: [1, H_kv, T_local, D] (strided views, e.g.
    the packed [T, H, D] layout permuted), the same shapes on every rank.
    Returns (out, lse): out like q (in out's dtype when given, else q's),
    lse float32 [1, H, T_local]."""
    import torch.distributed as dist
    W = dist.get_world_size(group)
    r = dist.get_rank(group)
    glob = (lambda i: dist.get_global_rank(group, i)) if group is not None else (lambda i: i)
    to_rank, from_rank = glob((r + 1) % W), glob((r - 1) % W)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    attn_fn = attn_fn or _lib_attn
    merge_fn = merge_fn or _lib_merge
    host = _host_exchange(q, group)
    if staging is None or not staging.fits(q, k, host):
        staging = RingStaging(q, k, host)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if W == 1:
        return attn_fn(q, k, v, scale, (out, lse))

    slot, other = 0, 1
    cur, nxt = staging.kv[slot], staging.kv[other]
    cur[0].copy_(k)
    cur[1].copy_(v)
    acc: Optional[Pair] = None
    for s in range(W):
        if host and staging.copied[other] is not None:
            # the host buffer about to be received into was last copied to the device
            # asynchronously: that copy must have read it first
            staging.copied[other].synchronize()
        # pass the chunk on while this step's attention runs (both only read it)
        reqs = []
        if s + 1 < W:
            reqs.append(dist.isend(cur, to_rank, group=group))
            reqs.append(dist.irecv(nxt, from_rank, group=group))
        if host:
            staging.kv_dev.copy_(cur, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record()
            staging.copied[slot] = ev
            kk, vv = staging.kv_dev[0], staging.kv_dev[1]
        else:
            kk, vv = cur[0], cur[1]
        part = attn_fn(q, kk, vv, scale, staging.parts[s % 2])
        if acc is None:
            acc = part
        else:
            last = s + 1 == W
            acc = merge_fn([acc[0], part[0]], [acc[1], part[1]], (out, lse) if last else staging.accs[s % 2])
        for req in reqs:
            req.wait()
        slot, other = other, slot
        cur, nxt = nxt, cur
    return acc
