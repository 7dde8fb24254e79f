"""CPU oracle for masked attention, LSE merge, paged KV append/gather and
paged GQA decode.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The library never imports
this package, and nothing here imports the library.  Everything is computed
in fp64 (attention and decode in plain C with OpenMP, ``attn_oracle.c``;
merge, append and gather in numpy), materialising every score row.

Sources, by page title and section:
* masked attention with an additive key-padding mask -- "MultiheadAttention
  fast path used 18 GB of VRAM" (TL;DR; measuring on the CPU; the mask
  direction note): padded keys get -inf added before the softmax.
* LSE output and merge -- "[sglang] ROCm aiter ring attention and K/V buffer
  reuse" (section 1, aiter.py): each chunk returns (out_i, lse_i) and the
  chunks combine as out = sum_i exp(lse_i - lse) * out_i; the packed path
  returns lse laid out [H, Tq].
* paged cache -- "LLM inference memory accounting" (section 15): a block table
  maps each logical block to a physical block; (section 10/11) KV bytes per
  token = layers x 2 x H_KV x D_head x B_elem.
* decode -- "KV cache in nanoVLM" (how KV caching optimises inference): the
  new token's K/V is appended to the cache and its query attends over it.
* INT8 KV -- "LLM inference memory accounting" (section 18): codes plus a
  float32 scale per token row; attention runs on the dequantised values.
* prefill -- "KV cache in nanoVLM" (prefill and decode phases) and "LLM
  inference memory accounting" (section 20, chunked prefill): a prompt or a
  chunk of it is processed in one pass, its K/V written to the cache; a
  causal query attends to no later position.

Every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle.py`` against brute force in arbitrary precision, a
library routine, closed forms, invariants and the pages' worked numbers.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import platform
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, f"liboracle_{platform.machine()}.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (-O2 -fopenmp, IEEE semantics kept)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_attn.restype = ctypes.c_int
            lib.oracle_attn.argtypes = [i64] * 6 + [p, ctypes.c_int, p] * 3 + [
                p, i64, ctypes.c_double, p, i64, p, p]
            lib.oracle_paged_decode.restype = ctypes.c_int
            lib.oracle_paged_decode.argtypes = [i64] * 6 + [p, ctypes.c_int, p, p, ctypes.c_int,
                                                           p, i64, i64, p, ctypes.c_double, p, p]
            lib.oracle_paged_prefill.restype = ctypes.c_int
            lib.oracle_paged_prefill.argtypes = [i64] * 7 + [p, ctypes.c_int, p, p, ctypes.c_int,
                                                            p, i64, i64, p, ctypes.c_int, ctypes.c_double, p, p]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _as_host(t):
    """(numpy array holding the raw elements, dtype code, element strides).

    bfloat16 tensors are passed as their 16-bit patterns; the C side widens
    them exactly."""
    import torch
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(t)
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        code = BF16
        arr = t.view(torch.int16)
    elif t.dtype == torch.float32:
        code = F32
        arr = t
    elif t.dtype == torch.float64:
        code = F32
        arr = t.to(torch.float32)
        if not torch.equal(arr.to(torch.float64), t):
            raise ValueError("oracle inputs must be exactly representable in float32")
    else:
        raise TypeError(f"oracle inputs must be float32 or bfloat16, got {t.dtype}")
    return arr, code


def attn(q, k, v, mask=None, scale: Optional[float] = None,
         rows: Optional[Sequence[int]] = None):
    """Masked attention over [B, Hq, Pq, D] / [B, Hkv, Pk, D] (any strides;
    keys and values are made contiguous along D).

    Returns ``(out, lse)`` as float64 numpy arrays: ``[B, Hq, Pq, D]`` and
    ``[B, Hq, Pq]`` when ``rows`` is None, else ``[len(rows), D]`` and
    ``[len(rows)]`` for the flat row ids ``(b * Hq + h) * Pq + i``."""
    import torch
    lib = _load()
    B, Hq, Pq, D = q.shape
    Bk, Hkv, Pk, Dk = k.shape
    assert Bk == B and Dk == D and tuple(v.shape) == tuple(k.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qa, qc = _as_host(q)
    ka, kc = _as_host(k)
    va, vc = _as_host(v)
    if ka.stride(3) != 1:
        ka = ka.contiguous()
    if va.stride(3) != 1:
        va = va.contiguous()
    qst = np.array(qa.stride(), dtype=np.int64)
    kst = np.array(ka.stride(), dtype=np.int64)
    vst = np.array(va.stride(), dtype=np.int64)
    if mask is not None:
        m = mask.detach().cpu().to(torch.float32)
        assert tuple(m.shape) == (B, Pk)
        m = m.contiguous()
        mptr, mstride = m.data_ptr(), m.stride(0)
    else:
        m, mptr, mstride = None, None, 0
    if rows is None:
        n = B * Hq * Pq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.size
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_attn(B, Hq, Hkv, Pq, Pk, D,
                         qa.data_ptr(), qc, qst.ctypes.data,
                         ka.data_ptr(), kc, kst.ctypes.data,
                         va.data_ptr(), vc, vst.ctypes.data,
                         mptr, mstride, float(scale),
                         None if rows_arr is None else rows_arr.ctypes.data, n,
                         out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn: bad arguments")
    if rows is None:
        return out.reshape(B, Hq, Pq, D), lse.reshape(B, Hq, Pq)
    return out, lse


def merge(outs: Sequence[np.ndarray], lses: Sequence[np.ndarray]):
    """Merge chunk results that each carry their softmax LSE.

    lse = M + log(sum_i exp(lse_i - M)) with M = max_i lse_i (stable form of
    log sum_i exp(lse_i)), and out = sum_i exp(lse_i - lse) * out_i -- the
    online-softmax merge of the ring-attention page (section 1).  Partials
    with lse_i = -inf (all keys masked) carry weight 0; if every partial is
    -inf the result is out = 0, lse = -inf.  Shapes: outs[i] [..., D],
    lses[i] [...]; returns float64 arrays."""
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = [np.asarray(l, dtype=np.float64) for l in lses]
    L = np.stack(lses)  # [n, ...]
    M = np.max(L, axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    with np.errstate(over="ignore", invalid="ignore"):
        w_unnorm = np.where(np.isneginf(L), 0.0, np.exp(L - Ms))
    tot = w_unnorm.sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(finite, Ms + np.log(np.where(finite, tot, 1.0)), -np.inf)
    out = np.zeros_like(outs[0])
    for i, o in enumerate(outs):
        with np.errstate(over="ignore", invalid="ignore"):
            w = np.where(finite & ~np.isneginf(L[i]), np.exp(L[i] - np.where(finite, lse, 0.0)), 0.0)
        out = out + w[..., None] * o
    return out, lse


def kv_append(k_cache, v_cache, block_table, pos, k_new, v_new, block_size: int = 16):
    """Expected caches after appending one token per sequence.

    For sequence b, the new token goes to physical block
    ``block_table[b, pos[b] // block_size]``, slot ``pos[b] % block_size``;
    every other slot is unchanged.  Works on the raw 16-bit patterns (bf16)
    or 32-bit patterns (f32), so the comparison is bit for bit.  Returns numpy
    copies of (k_cache, v_cache) viewed as integers."""
    kc = _bits(k_cache).copy()
    vc = _bits(v_cache).copy()
    bt = np.asarray(_np(block_table), dtype=np.int64)
    ps = np.asarray(_np(pos), dtype=np.int64)
    kn = _bits(k_new)
    vn = _bits(v_new)
    for b in range(ps.shape[0]):
        blk = bt[b, ps[b] // block_size]
        slot = ps[b] % block_size
        kc[blk, :, slot, :] = kn[b]
        vc[blk, :, slot, :] = vn[b]
    return kc, vc


def kv_append_chunk(k_cache, v_cache, block_table, start_pos, k_new, v_new, block_size: int = 16):
    """Expected caches after appending a chunk of T tokens per sequence.

    Token i of sequence b's chunk (``k_new[b, :, i]``, ``[B, Hkv, T, D]``) goes
    to position ``start_pos[b] + i``: physical block
    ``block_table[b, (start_pos[b] + i) // block_size]``, slot
    ``(start_pos[b] + i) % block_size``.  Bit patterns, like ``kv_append``."""
    kc = _bits(k_cache).copy()
    vc = _bits(v_cache).copy()
    bt = np.asarray(_np(block_table), dtype=np.int64)
    sp = np.asarray(_np(start_pos), dtype=np.int64)
    kn = _bits(k_new)
    vn = _bits(v_new)
    for b in range(sp.shape[0]):
        for i in range(kn.shape[2]):
            t = sp[b] + i
            blk = bt[b, t // block_size]
            kc[blk, :, t % block_size, :] = kn[b, :, i, :]
            vc[blk, :, t % block_size, :] = vn[b, :, i, :]
    return kc, vc


def paged_gather(cache, block_table, lens, block_size: int = 16):
    """Contiguous per-sequence K (or V) by walking the block table token by
    token: result[b] has shape [Hkv, lens[b], D] (raw integer bit patterns)."""
    c = _bits(cache)
    bt = np.asarray(_np(block_table), dtype=np.int64)
    out = []
    for b, L in enumerate(np.asarray(_np(lens), dtype=np.int64)):
        rows = []
        for t in range(int(L)):
            rows.append(c[bt[b, t // block_size], :, t % block_size, :])
        if rows:
            out.append(np.stack(rows, axis=1))
        else:
            out.append(np.zeros((c.shape[1], 0, c.shape[3]), dtype=c.dtype))
    return out


def paged_decode(q, k_cache, v_cache, block_table, ctx_lens, scale: Optional[float] = None,
                 block_size: int = 16):
    """One query token per sequence attending over its paged cache.

    q: [B, Hq, D]; caches [num_blocks, Hkv, block_size, D]; block_table int32
    [B, width]; ctx_lens int32 [B] (tokens attended, the appended one
    included).  Query head h reads KV head h // (Hq // Hkv).  Returns float64
    (out [B, Hq, D], lse [B, Hq])."""
    import torch
    lib = _load()
    B, Hq, D = q.shape
    nb, Hkv, bs, Dk = k_cache.shape
    assert bs == block_size and Dk == D
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qa, qc = _as_host(q.contiguous() if hasattr(q, "contiguous") else q)
    qa = qa.contiguous()  # held here: the C call reads it
    ka, kc = _as_host(k_cache.contiguous())
    va, vc = _as_host(v_cache.contiguous())
    assert kc == vc
    bt = torch.as_tensor(_np(block_table)).to(torch.int32).contiguous()
    cl = torch.as_tensor(_np(ctx_lens)).to(torch.int32).contiguous()
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = lib.oracle_paged_decode(B, Hq, Hkv, D, bs, nb, qa.data_ptr(), qc,
                                 ka.data_ptr(), va.data_ptr(), kc,
                                 bt.data_ptr(), bt.stride(0), bt.shape[1], cl.data_ptr(),
                                 float(scale), out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_paged_decode: block table entry outside the cache "
                         "or context longer than the table")
    return out, lse


def paged_prefill(q, k_cache, v_cache, block_table, start_pos, causal: bool, scale: Optional[float] = None,
                  block_size: int = 16):
    """A chunk of T query tokens per sequence attending over its paged cache.

    q: [B, Hq, T, D]; caches [num_blocks, Hkv, block_size, D] that already
    hold the chunk at positions ``start_pos[b] + i``; block_table int32
    [B, width]; start_pos int32 [B] (tokens cached before the chunk).  Query
    i attends over positions ``[0, start_pos[b] + i]`` when ``causal``, else
    over ``[0, start_pos[b] + T)``.  Returns float64 (out [B, Hq, T, D],
    lse [B, Hq, T])."""
    import torch
    lib = _load()
    B, Hq, T, D = q.shape
    nb, Hkv, bs, Dk = k_cache.shape
    assert bs == block_size and Dk == D
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qa, qc = _as_host(q.contiguous() if hasattr(q, "contiguous") else q)
    qa = qa.contiguous()  # held here: the C call reads it
    ka, kc = _as_host(k_cache.contiguous())
    va, vc = _as_host(v_cache.contiguous())
    assert kc == vc
    bt = torch.as_tensor(_np(block_table)).to(torch.int32).contiguous()
    sp = torch.as_tensor(_np(start_pos)).to(torch.int32).contiguous()
    out = np.zeros((B, Hq, T, D), dtype=np.float64)
    lse = np.zeros((B, Hq, T), dtype=np.float64)
    rc = lib.oracle_paged_prefill(B, Hq, Hkv, T, D, bs, nb, qa.data_ptr(), qc,
                                  ka.data_ptr(), va.data_ptr(), kc,
                                  bt.data_ptr(), bt.stride(0), bt.shape[1], sp.data_ptr(), int(bool(causal)),
                                  float(scale), out.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_paged_prefill: block table entry outside the cache "
                         "or sequence longer than the table")
    return out, lse


# --------------------------------------------------------------------------
# INT8 KV ("LLM inference memory accounting", section 18: BF16 KV to INT8
# halves the payload and adds scale metadata and a dequantisation step)
# --------------------------------------------------------------------------
def quantize_rows_q8(x):
    """Symmetric INT8 code of each row (last axis) with one float32 scale per
    row, every step in float32 as written:
        a     = max_d |x_d|
        scale = a / 127                      (0 for an all-zero row)
        q_d   = clamp(rint(x_d / scale), -127, 127)   (0 when scale is 0)
    rint rounds half to even.  Returns (int8 codes, float32 scales)."""
    import torch
    xs = np.asarray(x.detach().cpu().to(torch.float32).numpy() if hasattr(x, "detach") else x, dtype=np.float32)
    a = np.max(np.abs(xs), axis=-1)
    scale = (a / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    q = np.rint(xs / safe[..., None]).astype(np.float32)
    q = np.clip(q, -127, 127)
    q = np.where(scale[..., None] > 0, q, 0).astype(np.int8)
    return q, scale


def dequantize_rows_q8(q, scale):
    """x_hat = q * scale in float32 (exact in float64 afterwards)."""
    return (np.asarray(q, dtype=np.float32) * np.asarray(scale, dtype=np.float32)[..., None]).astype(np.float32)


def kv_append_q8(kq_cache, vq_cache, k_scale, v_scale, block_table, pos, k_new, v_new, block_size: int = 16):
    """Expected INT8 caches after appending one token per sequence: the new
    token's K and V rows (per KV head) are quantised with quantize_rows_q8 and
    written, codes and scales, to block block_table[b, pos // block_size],
    slot pos % block_size; pos < 0 skips the sequence.  Caches
    [num_blocks, Hkv, block_size, D] int8, scales [num_blocks, Hkv,
    block_size] float32.  Returns numpy copies (kq, vq, k_scale, v_scale)."""
    kq = np.array(_np(kq_cache), dtype=np.int8, copy=True)
    vq = np.array(_np(vq_cache), dtype=np.int8, copy=True)
    ks = np.array(_np(k_scale), dtype=np.float32, copy=True)
    vs = np.array(_np(v_scale), dtype=np.float32, copy=True)
    bt = np.asarray(_np(block_table), dtype=np.int64)
    ps = np.asarray(_np(pos), dtype=np.int64)
    qk, sk = quantize_rows_q8(k_new)
    qv, sv = quantize_rows_q8(v_new)
    for b in range(ps.shape[0]):
        if ps[b] < 0:
            continue
        blk = bt[b, ps[b] // block_size]
        slot = ps[b] % block_size
        kq[blk, :, slot, :] = qk[b]
        vq[blk, :, slot, :] = qv[b]
        ks[blk, :, slot] = sk[b]
        vs[blk, :, slot] = sv[b]
    return kq, vq, ks, vs


def paged_decode_q8(q, kq_cache, vq_cache, k_scale, v_scale, block_table, ctx_lens, scale: Optional[float] = None,
                    block_size: int = 16):
    """Paged decode over an INT8 cache: the definition of paged_decode applied
    to the dequantised K and V (q * scale, float32, exact in float64)."""
    import torch
    kd = torch.from_numpy(dequantize_rows_q8(_np(kq_cache), _np(k_scale)))
    vd = torch.from_numpy(dequantize_rows_q8(_np(vq_cache), _np(v_scale)))
    return paged_decode(q, kd, vd, block_table, ctx_lens, scale, block_size)


# --------------------------------------------------------------------------
# Memory arithmetic from the pages
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ModelShape:
    """KV sizing of a dense decoder ("LLM inference memory accounting",
    sections 10-11): bytes per token = layers x 2 (K and V) x KV heads x
    head dim x element bytes.  GQA/MQA enter through ``kv_heads``."""
    layers: int
    kv_heads: int
    head_dim: int
    kv_bytes: float

    def kv_bytes_per_token(self) -> float:
        return self.layers * 2 * self.kv_heads * self.head_dim * self.kv_bytes

    def sequence_kv_bytes(self, tokens: int) -> float:
        return self.kv_bytes_per_token() * tokens


def token_capacity(pool_bytes: int, bytes_per_token: int) -> int:
    """Physical KV tokens a pool holds, floor(M_pool / b_token) (same page,
    section 27)."""
    return int(pool_bytes // bytes_per_token)


def score_matrix_bytes(heads: int, P: int, elem_bytes: int) -> int:
    """Bytes of a materialised heads x P x P score matrix -- the buffer the
    MultiheadAttention fast path builds when a mask is passed."""
    return heads * P * P * elem_bytes


# --------------------------------------------------------------------------
def _np(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().numpy()
    return np.asarray(x)


def _bits(x):
    """Raw integer bit patterns of a bf16/f32 tensor (or integer array)."""
    import torch
    if isinstance(x, np.ndarray):
        return x
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy()
    if x.dtype == torch.float32:
        return x.view(torch.int32).numpy()
    return x.numpy()
