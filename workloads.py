"""Seeded synthetic inputs shaped like the workloads on the pages.

This module draws tensors and builds index structures; it holds none of the
attention arithmetic. Both sides of every parity check (the CUDA library and
the CPU oracle) and the benchmark take their inputs from here, generated on
the CPU from ``torch.Generator('cpu').manual_seed(seed)`` in a fixed order:

* attention: ``n_pad`` (only when the padded tail is random), then q, k, v.
  Values are float32 N(0, 1), cast to the config's dtype afterwards; the
  oracle receives the cast values (bf16 -> fp64 is exact).
* key-padding mask: additive float32 ``[B, Pk]``; 0 for a real key and -inf
  for a padded one (the decoder on the first page turns its boolean padding
  mask into exactly this form).
* paged decode: context lengths, the block permutation, the K cache, the V
  cache, k_new, v_new, q.  Every cache slot that holds no token of the
  context is NaN, so a kernel that reads a slot it should not read returns
  NaN instead of a plausible number.

The workloads themselves (sizes, dtypes, mask tails, the GQA decode shape)
follow the configurations named in ``ATTN_CONFIGS`` and ``DECODE_CONFIGS``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

NEG_INF = float("-inf")


# --------------------------------------------------------------------------
# Attention (prefill / patch self-attention / chunked attention)
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class AttnConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Pq: int
    Pk: int
    D: int
    dtype: torch.dtype
    # padded key tail: ("fixed", n) pads the last n keys of every batch row;
    # ("random", hi) draws n_pad uniformly from [0, hi] (inclusive) from the
    # seed, once, for all batch rows; ("none", 0) passes no mask at all.
    pad: tuple = ("none", 0)
    packed: bool = False  # tensors stored [T, H, D] (one sequence, B == 1)
    chunks: int = 1  # number of contiguous KV chunks merged through the LSE
    scale: Optional[float] = None  # default 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    def chunk_bounds(self) -> list[tuple[int, int]]:
        """Contiguous, equal KV chunks ``[lo, hi)`` (the last takes any rest)."""
        step = self.Pk // self.chunks
        out = []
        for c in range(self.chunks):
            lo = c * step
            hi = self.Pk if c == self.chunks - 1 else (c + 1) * step
            out.append((lo, hi))
        return out


ATTN_CONFIGS = {
    # tiny masked self-attention at the size the oracle checks in full
    "tiny_f32": AttnConfig("tiny_f32", 1, 16, 16, 512, 512, 64, torch.float32,
                           pad=("fixed", 37), scale=1.0 / 8.0),
    # patch self-attention of a 0.5 MP image: P = 1944 patches, 16 heads
    "patch_small": AttnConfig("patch_small", 1, 16, 16, 1944, 1944, 64, torch.bfloat16,
                              pad=("random", 64), scale=1.0 / 8.0),
    # packed [T, H, D] attention over two KV chunks merged through the LSE
    "chunked": AttnConfig("chunked", 1, 24, 24, 32760, 32760, 128, torch.bfloat16,
                          pad=("none", 0), packed=True, chunks=2),
    # patch self-attention of an 8 MP image: P = 32000, last 128 keys padded
    "patch_large": AttnConfig("patch_large", 1, 16, 16, 32000, 32000, 64, torch.bfloat16,
                              pad=("fixed", 128), scale=1.0 / 8.0),
}


@dataclasses.dataclass
class AttnInputs:
    cfg: AttnConfig
    q: torch.Tensor  # [B, Hq, Pq, D] (a strided view when packed)
    k: torch.Tensor  # [B, Hkv, Pk, D]
    v: torch.Tensor  # [B, Hkv, Pk, D]
    mask: Optional[torch.Tensor]  # [B, Pk] float32 additive, or None
    n_pad: int
    scale: float
    packed_q: Optional[torch.Tensor] = None  # [T, H, D] storage when packed
    packed_k: Optional[torch.Tensor] = None
    packed_v: Optional[torch.Tensor] = None


def _randn(shape, g, dtype) -> torch.Tensor:
    """N(0,1) float32 draws cast to ``dtype``, drawn in slabs along dim 0 so
    that large tensors never need a full float32 copy in host memory."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=dtype)
    if len(shape) == 0 or shape[0] == 0:
        return out
    per_row = max(1, math.prod(shape[1:]))
    rows = max(1, (1 << 24) // per_row)
    for lo in range(0, shape[0], rows):
        hi = min(shape[0], lo + rows)
        out[lo:hi] = torch.randn((hi - lo,) + shape[1:], generator=g, dtype=torch.float32).to(dtype)
    return out


def padding_mask(B: int, Pk: int, n_pad: Sequence[int] | int) -> torch.Tensor:
    """Additive key-padding mask: 0 for real keys, -inf for the padded tail."""
    m = torch.zeros(B, Pk, dtype=torch.float32)
    pads = [n_pad] * B if isinstance(n_pad, int) else list(n_pad)
    for b, n in enumerate(pads):
        if n > 0:
            m[b, Pk - n:] = NEG_INF
    return m


def make_attn_inputs(cfg: AttnConfig, seed: int = 0) -> AttnInputs:
    g = torch.Generator(device="cpu").manual_seed(seed)
    kind, val = cfg.pad
    if kind == "random":
        n_pad = int(torch.randint(0, val + 1, (1,), generator=g).item())
    elif kind == "fixed":
        n_pad = int(val)
    else:
        n_pad = 0
    if cfg.packed:
        assert cfg.B == 1
        pq = _randn((cfg.Pq, cfg.Hq, cfg.D), g, cfg.dtype)
        pk = _randn((cfg.Pk, cfg.Hkv, cfg.D), g, cfg.dtype)
        pv = _randn((cfg.Pk, cfg.Hkv, cfg.D), g, cfg.dtype)
        q = pq.permute(1, 0, 2).unsqueeze(0)
        k = pk.permute(1, 0, 2).unsqueeze(0)
        v = pv.permute(1, 0, 2).unsqueeze(0)
    else:
        pq = pk = pv = None
        q = _randn((cfg.B, cfg.Hq, cfg.Pq, cfg.D), g, cfg.dtype)
        k = _randn((cfg.B, cfg.Hkv, cfg.Pk, cfg.D), g, cfg.dtype)
        v = _randn((cfg.B, cfg.Hkv, cfg.Pk, cfg.D), g, cfg.dtype)
    mask = padding_mask(cfg.B, cfg.Pk, n_pad) if kind != "none" else None
    return AttnInputs(cfg, q, k, v, mask, n_pad, cfg.softmax_scale, pq, pk, pv)


def make_attn(B, Hq, Hkv, Pq, Pk, D, dtype=torch.bfloat16, n_pad=0, seed=0,
              with_mask=True, packed=False) -> AttnInputs:
    """Free-form attention inputs for parity cases at other sizes.

    ``n_pad`` may be an int (same tail for every batch row) or a list with
    one tail length per batch row."""
    cfg = AttnConfig("custom", B, Hq, Hkv, Pq, Pk, D, dtype,
                     pad=("fixed", 0) if with_mask else ("none", 0), packed=packed)
    inp = make_attn_inputs(cfg, seed)
    if with_mask:
        inp.mask = padding_mask(B, Pk, n_pad)
        inp.n_pad = n_pad if isinstance(n_pad, int) else max(n_pad)
    return inp


def attn_flops(B, Hq, Pq, Pk_valid, D) -> float:
    """Algorithmic FLOPs of attention over the valid keys: QK^T and PV, each
    2*Pq*Pk*D per head (multiply and add counted separately)."""
    return 4.0 * B * Hq * Pq * Pk_valid * D


# --------------------------------------------------------------------------
# Paged GQA decode
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    ctx_lo: int  # context length before the append, inclusive range
    ctx_hi: int
    spare_blocks: int
    scale: Optional[float] = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def max_blocks(self) -> int:
        """Block-table width: enough blocks for the longest context plus the
        appended token."""
        return -(-(self.ctx_hi + 1) // self.block_size)


DECODE_CONFIGS = {
    # 64 sequences, 32 query heads sharing 8 KV heads, head dim 128,
    # 16-token blocks, contexts uniform in [512, 8192] before the append
    "decode": DecodeConfig("decode", 64, 32, 8, 128, 16, 512, 8192, 64),
}


@dataclasses.dataclass
class DecodeInputs:
    cfg: DecodeConfig
    ctx: torch.Tensor  # int32 [B]: tokens in the cache before the append
    pos: torch.Tensor  # int32 [B]: slot index the new token goes to (== ctx)
    ctx_lens: torch.Tensor  # int32 [B]: tokens attended after the append (ctx + 1)
    block_table: torch.Tensor  # int32 [B, max_blocks]; unused entries are -1
    k_cache: torch.Tensor  # bf16 [num_blocks, Hkv, block_size, D]
    v_cache: torch.Tensor
    k_new: torch.Tensor  # bf16 [B, Hkv, D]
    v_new: torch.Tensor
    q: torch.Tensor  # bf16 [B, Hq, D]
    scale: float

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])


def make_decode_inputs(cfg: DecodeConfig, seed: int = 0,
                       ctx: Optional[Sequence[int]] = None,
                       dtype: torch.dtype = torch.bfloat16) -> DecodeInputs:
    """Paged-cache decode step inputs.

    ``ctx`` overrides the drawn context lengths (edge cases); otherwise they
    are uniform integers in ``[ctx_lo, ctx_hi]``. Each sequence owns
    ``ceil((ctx + 1) / block_size)`` physical blocks taken from one seeded
    random permutation of all physical blocks, in order; ``spare_blocks``
    extra physical blocks belong to no sequence."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    B, bs = cfg.B, cfg.block_size
    if ctx is None:
        ctx_t = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (B,), generator=g)
    else:
        ctx_t = torch.tensor(list(ctx), dtype=torch.int64)
        assert ctx_t.numel() == B
    lens = ctx_t + 1
    nblk = (lens + bs - 1) // bs
    width = max(cfg.max_blocks, int(nblk.max().item()))
    n_phys = int(nblk.sum().item()) + cfg.spare_blocks
    perm = torch.randperm(n_phys, generator=g)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    k_cache = _randn((n_phys, cfg.Hkv, bs, cfg.D), g, dtype)
    v_cache = _randn((n_phys, cfg.Hkv, bs, cfg.D), g, dtype)
    # every slot not holding one of the first ctx tokens of its sequence is NaN
    filled = torch.zeros(n_phys, bs, dtype=torch.bool)
    for b in range(B):
        t = torch.arange(int(ctx_t[b]))
        filled[bt[b, (t // bs)].long(), t % bs] = True
    hole = ~filled
    k_cache.permute(0, 2, 1, 3)[hole] = float("nan")
    v_cache.permute(0, 2, 1, 3)[hole] = float("nan")
    k_new = _randn((B, cfg.Hkv, cfg.D), g, dtype)
    v_new = _randn((B, cfg.Hkv, cfg.D), g, dtype)
    q = _randn((B, cfg.Hq, cfg.D), g, dtype)
    return DecodeInputs(cfg, ctx_t.to(torch.int32), ctx_t.to(torch.int32),
                        lens.to(torch.int32), bt, k_cache, v_cache, k_new, v_new, q,
                        cfg.softmax_scale)


def decode_kv_bytes(ctx_lens: torch.Tensor, Hkv: int, D: int, elem_bytes: int = 2) -> int:
    """Algorithmic KV bytes one decode step reads: K and V of every attended
    token of every KV head."""
    return int(ctx_lens.to(torch.int64).sum().item()) * 2 * Hkv * D * elem_bytes


# --------------------------------------------------------------------------
# Paged (chunked) prefill
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T: int  # chunk tokens per sequence
    block_size: int
    start_lo: int  # tokens cached before the chunk, inclusive range
    start_hi: int
    spare_blocks: int
    causal: bool = True
    scale: Optional[float] = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)


PREFILL_CONFIGS = {
    # the decode workload's model shape (32 query heads on 8 KV heads, D 128,
    # 16-token blocks); 16 sequences each prefilling a 1024-token chunk after
    # 0..7168 cached tokens
    "prefill_chunk": PrefillConfig("prefill_chunk", 16, 32, 8, 128, 1024, 16, 0, 7168, 16),
}


@dataclasses.dataclass
class PrefillInputs:
    cfg: PrefillConfig
    start_pos: torch.Tensor  # int32 [B]: tokens cached before the chunk
    block_table: torch.Tensor  # int32 [B, width]; unused entries are -1
    k_cache: torch.Tensor  # [num_blocks, Hkv, block_size, D]; NaN where nothing is cached
    v_cache: torch.Tensor
    k_new: torch.Tensor  # [B, Hkv, T, D]: the chunk's keys and values
    v_new: torch.Tensor
    q: torch.Tensor  # [B, Hq, T, D]
    scale: float

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def make_prefill_inputs(cfg: PrefillConfig, seed: int = 0, start: Optional[Sequence[int]] = None,
                        dtype: torch.dtype = torch.bfloat16) -> PrefillInputs:
    """Paged-cache prefill inputs: ``start`` (drawn uniform in
    ``[start_lo, start_hi]`` unless given) tokens are cached per sequence and
    a chunk of ``T`` follows.  Each sequence owns ``ceil((start + T) /
    block_size)`` physical blocks from one seeded random permutation;
    unfilled slots hold NaN, so reading one shows."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    B, bs, T = cfg.B, cfg.block_size, cfg.T
    if start is None:
        st = torch.randint(cfg.start_lo, cfg.start_hi + 1, (B,), generator=g)
    else:
        st = torch.tensor(list(start), dtype=torch.int64)
        assert st.numel() == B
    total = st + T
    nblk = (total + bs - 1) // bs
    width = int(nblk.max().item()) if B > 0 else 1
    n_phys = int(nblk.sum().item()) + cfg.spare_blocks
    perm = torch.randperm(n_phys, generator=g)
    bt = torch.full((B, max(width, 1)), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    k_cache = _randn((n_phys, cfg.Hkv, bs, cfg.D), g, dtype)
    v_cache = _randn((n_phys, cfg.Hkv, bs, cfg.D), g, dtype)
    filled = torch.zeros(n_phys, bs, dtype=torch.bool)
    for b in range(B):
        t = torch.arange(int(st[b]))
        filled[bt[b, (t // bs)].long(), t % bs] = True
    k_cache.permute(0, 2, 1, 3)[~filled] = float("nan")
    v_cache.permute(0, 2, 1, 3)[~filled] = float("nan")
    k_new = _randn((B, cfg.Hkv, T, cfg.D), g, dtype)
    v_new = _randn((B, cfg.Hkv, T, cfg.D), g, dtype)
    q = _randn((B, cfg.Hq, T, cfg.D), g, dtype)
    return PrefillInputs(cfg, st.to(torch.int32), bt, k_cache, v_cache, k_new, v_new, q, cfg.softmax_scale)


def prefill_flops(start_pos: torch.Tensor, T: int, Hq: int, D: int, causal: bool) -> float:
    """Algorithmic FLOPs of a prefill chunk: 4*D per (query, attended key)
    per head; query i of a causal chunk attends start + i + 1 keys."""
    st = start_pos.to(torch.float64)
    if causal:
        keys = (st * T + T * (T + 1) / 2).sum().item()
    else:
        keys = ((st + T) * T).sum().item()
    return 4.0 * Hq * D * keys


# --------------------------------------------------------------------------
# Paged decode over an INT8 cache (codes and one float32 scale per token row)
# --------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeInputsQ8:
    cfg: DecodeConfig
    ctx: torch.Tensor
    pos: torch.Tensor
    ctx_lens: torch.Tensor
    block_table: torch.Tensor
    kq_cache: torch.Tensor  # int8 [num_blocks, Hkv, block_size, D]; 0 in unfilled slots
    vq_cache: torch.Tensor
    k_scale: torch.Tensor  # float32 [num_blocks, Hkv, block_size]; NaN in unfilled slots
    v_scale: torch.Tensor
    k_new: torch.Tensor  # bf16 [B, Hkv, D]
    v_new: torch.Tensor
    q: torch.Tensor  # bf16 [B, Hq, D]
    scale: float

    @property
    def num_blocks(self) -> int:
        return int(self.kq_cache.shape[0])


def make_decode_inputs_q8(cfg: DecodeConfig, seed: int = 0, ctx: Optional[Sequence[int]] = None) -> DecodeInputsQ8:
    """The decode workload's shapes and block assignment with an INT8 cache:
    codes uniform in [-127, 127] and scales uniform in [0.01, 0.04] (rows of
    N(0,1)-sized values) for slots holding one of the first ctx tokens; codes
    0 and scale NaN everywhere else, so reading an unfilled slot shows."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    B, bs = cfg.B, cfg.block_size
    if ctx is None:
        ctx_t = torch.randint(cfg.ctx_lo, cfg.ctx_hi + 1, (B,), generator=g)
    else:
        ctx_t = torch.tensor(list(ctx), dtype=torch.int64)
        assert ctx_t.numel() == B
    lens = ctx_t + 1
    nblk = (lens + bs - 1) // bs
    width = max(cfg.max_blocks, int(nblk.max().item()))
    n_phys = int(nblk.sum().item()) + cfg.spare_blocks
    perm = torch.randperm(n_phys, generator=g)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    shape = (n_phys, cfg.Hkv, bs, cfg.D)
    kq = torch.randint(-127, 128, shape, generator=g, dtype=torch.int32).to(torch.int8)
    vq = torch.randint(-127, 128, shape, generator=g, dtype=torch.int32).to(torch.int8)
    ks = 0.01 + 0.03 * torch.rand((n_phys, cfg.Hkv, bs), generator=g)
    vs = 0.01 + 0.03 * torch.rand((n_phys, cfg.Hkv, bs), generator=g)
    filled = torch.zeros(n_phys, bs, dtype=torch.bool)
    for b in range(B):
        t = torch.arange(int(ctx_t[b]))
        filled[bt[b, (t // bs)].long(), t % bs] = True
    hole = ~filled
    kq.permute(0, 2, 1, 3)[hole] = 0
    vq.permute(0, 2, 1, 3)[hole] = 0
    ks.permute(0, 2, 1)[hole] = float("nan")
    vs.permute(0, 2, 1)[hole] = float("nan")
    k_new = _randn((B, cfg.Hkv, cfg.D), g, torch.bfloat16)
    v_new = _randn((B, cfg.Hkv, cfg.D), g, torch.bfloat16)
    q = _randn((B, cfg.Hq, cfg.D), g, torch.bfloat16)
    return DecodeInputsQ8(cfg, ctx_t.to(torch.int32), ctx_t.to(torch.int32), lens.to(torch.int32), bt, kq, vq,
                          ks.to(torch.float32), vs.to(torch.float32), k_new, v_new, q, cfg.softmax_scale)


def decode_kv_bytes_q8(ctx_lens: torch.Tensor, Hkv: int, D: int) -> int:
    """Algorithmic KV bytes of one INT8 decode step: codes of K and V plus
    their two float32 row scales, for every attended token of every KV head."""
    return int(ctx_lens.to(torch.int64).sum().item()) * Hkv * (2 * D + 8)
