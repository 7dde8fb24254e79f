"""Python binding of libattn (masked attention with LSE, LSE merge, paged KV
append, paged GQA decode) for one GB300 GPU.

This module only marshals arguments: it turns torch tensors into the C ABI's
pointer/shape/stride descriptors (``include/libattn.h``) and calls the shared
library through ctypes on the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; torch supplies device memory
(outputs and workspaces the caller did not pass are allocated with it) and
the stream.  There is no CPU fallback: if the library is missing or a call
fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

import torch

from . import build as _build

__all__ = [
    "load", "LibAttnError", "Workspace",
    "attn_fwd", "attn_lse_merge", "kv_append", "paged_decode_attn", "paged_kv_gather",
    "attn_fwd_workspace_size", "paged_decode_workspace_size", "check_device_status",
]

ATTN_F32, ATTN_BF16 = 0, 1
_STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
           4: "ATTN_ERR_TIMEOUT", 5: "ATTN_ERR_DEVICE_BOUNDS", 6: "ATTN_ERR_WORKSPACE"}


class LibAttnError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call}: {_STATUS.get(status, status)}")


class AttnTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class AttnKVCache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class AttnKVCacheQ8(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("reserved", ctypes.c_int32)]


def _signatures() -> dict:
    """ctypes result and argument types of every libattn entry point."""
    P, I32, I64, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    T = ctypes.POINTER(AttnTensor)
    C = ctypes.POINTER(AttnKVCache)
    CQ = ctypes.POINTER(AttnKVCacheQ8)
    return {
        "attn_version": (I32, []),
        "attn_status_string": (ctypes.c_char_p, [I32]),
        "attn_fwd_workspace_size": (SZ, []),
        "attn_fwd_workspace_size_for": (SZ, [I32, I32, I64, I32]),
        "kv_append_workspace_size": (SZ, []),
        "paged_decode_workspace_size": (SZ, [I32, I32, I32, I32, I32]),
        "attn_fwd": (I32, [T, T, T, P, I64, F, T, P, P, SZ, P]),
        "attn_fwd_varlen": (I32, [T, T, T, P, F, T, P, P, SZ, P]),
        "attn_key_padding_to_additive": (I32, [P, I64, I32, I64, P, I64, P]),
        "attn_lse_merge": (I32, [I32, T, ctypes.POINTER(P), T, P, P]),
        "kv_append": (I32, [C, P, I64, I32, P, T, T, P, SZ, P]),
        "paged_decode_attn": (I32, [T, C, P, I64, I32, P, F, T, P, P, SZ, P]),
        "paged_decode_attn_append": (I32, [T, T, T, C, P, I64, I32, P, F, T, P, P, SZ, P]),
        "paged_prefill_attn": (I32, [T, T, T, C, P, I64, I32, P, I32, F, T, P, P, SZ, P]),
        "kv_append_q8": (I32, [CQ, P, I64, I32, P, T, T, P, SZ, P]),
        "paged_decode_attn_q8": (I32, [T, CQ, P, I64, I32, P, F, T, P, P, SZ, P]),
        "paged_decode_attn_append_q8": (I32, [T, T, T, CQ, P, I64, I32, P, F, T, P, P, SZ, P]),
        "paged_kv_gather": (I32, [C, I32, P, I64, I32, P, I32, I64, P, P, SZ, P]),
        "paged_decode_attn_noalloc": (I32, [T, C, P, I64, I32, P, F, T, P, P, P]),
        "attn_check_device_status": (I32, [P, ctypes.POINTER(ctypes.c_uint32), P]),
        "attn_reset_device_status": (I32, [P, P]),
        "attn_selftest_wait_timeout": (I32, [P, SZ, ctypes.c_uint32, P]),
    }


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load libattn.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"libattn is not built ({path} missing); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            _build.build()
        lib = ctypes.CDLL(path)
        sig = _signatures()
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def exported_symbols() -> list[str]:
    return ["attn_fwd", "attn_lse_merge", "kv_append", "paged_decode_attn", "paged_kv_gather",
            "attn_fwd_workspace_size", "kv_append_workspace_size", "paged_decode_workspace_size",
            "attn_check_device_status", "attn_reset_device_status", "attn_status_string", "attn_version",
            "paged_decode_attn_noalloc", "attn_selftest_wait_timeout", "attn_fwd_varlen",
            "attn_key_padding_to_additive", "paged_decode_attn_append", "paged_prefill_attn",
            "attn_fwd_workspace_size_for", "kv_append_q8", "paged_decode_attn_q8", "paged_decode_attn_append_q8"]


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"libattn takes bfloat16 or float32 tensors, got {t.dtype}")


def _desc(t: torch.Tensor) -> AttnTensor:
    if not _on_device(t):
        raise ValueError("libattn tensors must be on a CUDA device")
    d = AttnTensor()
    d.data = t.data_ptr()
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return d


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(name: str, st: int):
    if st != 0:
        raise LibAttnError(name, st)


# Arguments that reach the library as bare pointers (LSE buffers, masks,
# block tables, per-sequence positions and lengths) carry no shape the C side
# could check, so their dtype, layout and size are checked here, with real
# exceptions rather than asserts (which `python -O` would drop, leaving a
# kernel to read or write past a short buffer), and their device when the
# pointer is taken.
def _require(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _on_device(t: torch.Tensor) -> bool:
    """Whether t lives where the library's kernels can read it."""
    return t.is_cuda


def _ptr(t: Optional[torch.Tensor], name: str = "tensor"):
    """Device pointer of t (None passes through as NULL)."""
    if t is None:
        return None
    _require(_on_device(t), f"{name} must be on a CUDA device")
    return t.data_ptr()


def _check_f32_buffer(t: torch.Tensor, numel: int, name: str):
    """float32, contiguous, exactly `numel` elements."""
    _require(isinstance(t, torch.Tensor), f"{name} must be a torch tensor")
    _require(t.dtype == torch.float32, f"{name} must be float32, got {t.dtype}")
    _require(t.is_contiguous(), f"{name} must be contiguous")
    _require(t.numel() == numel, f"{name} must hold {numel} elements, got {t.numel()}")


def _check_int32_vec(t: torch.Tensor, n: int, name: str):
    """int32 [n], contiguous."""
    _require(isinstance(t, torch.Tensor), f"{name} must be a torch tensor")
    _require(t.dtype == torch.int32, f"{name} must be int32, got {t.dtype}")
    _require(t.dim() == 1 and t.shape[0] == n and t.is_contiguous(), f"{name} must be contiguous [{n}], got "
             f"{tuple(t.shape)}")


def _check_block_table(t: torch.Tensor, batch: int):
    """int32 [>= batch, max_blocks] with unit stride along a row."""
    _require(isinstance(t, torch.Tensor), "block_table must be a torch tensor")
    _require(t.dtype == torch.int32, f"block_table must be int32, got {t.dtype}")
    _require(t.dim() == 2 and t.shape[0] >= batch and t.stride(1) == 1 and t.stride(0) >= t.shape[1],
             f"block_table must be [>= {batch}, max_blocks] with contiguous rows, got {tuple(t.shape)} "
             f"strides {tuple(t.stride())}")


class Workspace:
    """A zero-initialised device buffer for the library's workspace argument
    (its first word is the sticky device status)."""

    def __init__(self, nbytes: int, device=None):
        nbytes = max(256, (int(nbytes) + 255) // 256 * 256)
        self.tensor = torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")
        self.nbytes = nbytes

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()

    def status(self, stream=None) -> int:
        return check_device_status(self, stream)

    def reset(self, stream=None):
        _check("attn_reset_device_status", load().attn_reset_device_status(self.ptr, _stream(stream)))


_default_ws: dict = {}


def _small_ws(device) -> Workspace:
    key = torch.device(device).index
    ws = _default_ws.get(key)
    if ws is None:
        ws = Workspace(256, device=device)
        _default_ws[key] = ws
    return ws


def _attn_ws(q: torch.Tensor, k: torch.Tensor) -> Workspace:
    """Default attn_fwd workspace: the status word plus room for the per-tile
    key bounds and the last-wave partials of this shape (kept per device,
    grown when a call needs more).  It is shared by every call on the device
    that passes no workspace, so calls that may run concurrently (on
    different streams) must each pass their own."""
    need = attn_fwd_workspace_size_for(k.shape[0], k.shape[1], k.shape[2], k.shape[3])
    key = ("attn", torch.device(q.device).index)
    ws = _default_ws.get(key)
    if ws is None or ws.nbytes < need:
        ws = Workspace(max(need, 256), device=q.device)
        _default_ws[key] = ws
    return ws


def check_device_status(ws: Workspace, stream=None) -> int:
    raw = ctypes.c_uint32(0)
    st = load().attn_check_device_status(ws.ptr, ctypes.byref(raw), _stream(stream))
    return int(st)


def attn_fwd_workspace_size() -> int:
    return int(load().attn_fwd_workspace_size())


def attn_fwd_workspace_size_for(batch: int, kv_heads: int, num_keys: int, head_dim: int) -> int:
    return int(load().attn_fwd_workspace_size_for(batch, kv_heads, num_keys, head_dim))


def paged_decode_workspace_size(batch: int, num_q_heads: int, max_blocks: int, block_size: int = 16,
                                head_dim: int = 128) -> int:
    return int(load().paged_decode_workspace_size(batch, num_q_heads, max_blocks, block_size, head_dim))


# --------------------------------------------------------------------------
# the four calls
# --------------------------------------------------------------------------
def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, key_pad_mask: Optional[torch.Tensor] = None,
             scale: Optional[float] = None, out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             return_lse: bool = True, workspace: Optional[Workspace] = None, stream=None):
    """Masked exact attention; q [B, Hq, Pq, D], k/v [B, Hkv, Pk, D] (any
    strides with a contiguous last dim, e.g. packed [T, H, D] permuted to
    [1, H, T, D]).  key_pad_mask: float32 [B, Pk] additive (0 / -inf).
    Returns (out, lse) with lse float32 [B, Hq, Pq] (or out alone)."""
    lib = load()
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, q.shape[0] * q.shape[1] * q.shape[2], "lse")
    mptr, mstride = None, 0
    if key_pad_mask is not None:
        m = key_pad_mask
        _require(m.dtype == torch.float32, f"key_pad_mask must be float32 (additive), got {m.dtype}")
        _require(m.dim() == 2 and tuple(m.shape) == (q.shape[0], k.shape[2]) and m.stride(1) == 1,
                 f"key_pad_mask must be [{q.shape[0]}, {k.shape[2]}] with contiguous rows, got {tuple(m.shape)}")
        mptr, mstride = _ptr(m, "key_pad_mask"), m.stride(0)
    ws = workspace or _attn_ws(q, k)
    dq, dk, dv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    st = lib.attn_fwd(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), mptr, mstride, float(scale),
                      ctypes.byref(do), _ptr(lse, "lse"), ws.ptr, ws.nbytes, _stream(stream))
    _check("attn_fwd", st)
    return (out, lse) if return_lse else out


def attn_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, key_lens: torch.Tensor,
                    scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                    workspace: Optional[Workspace] = None, stream=None):
    """attn_fwd where batch row b attends to its first key_lens[b] keys (int32
    [B] on the device); KV tiles past the length are skipped."""
    lib = load()
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    _check_int32_vec(key_lens, q.shape[0], "key_lens")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, q.shape[0] * q.shape[1] * q.shape[2], "lse")
    ws = workspace or _attn_ws(q, k)
    dq, dk, dv, do = _desc(q), _desc(k), _desc(v), _desc(out)
    st = lib.attn_fwd_varlen(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), _ptr(key_lens, "key_lens"),
                             float(scale), ctypes.byref(do), _ptr(lse, "lse"), ws.ptr, ws.nbytes, _stream(stream))
    _check("attn_fwd_varlen", st)
    return (out, lse) if return_lse else out


def key_padding_to_additive(key_padding_mask: torch.Tensor, out: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """Boolean [B, Pk] key_padding_mask (True = padded key, the
    nn.MultiheadAttention convention) -> float32 additive mask (-inf / 0)."""
    lib = load()
    kpm = key_padding_mask
    _require(kpm.dim() == 2 and kpm.stride(1) == 1, "key_padding_mask must be [B, Pk] with contiguous rows")
    if kpm.dtype == torch.bool:
        kpm = kpm.view(torch.uint8)
    _require(kpm.dtype == torch.uint8, f"key_padding_mask must be bool or uint8, got {kpm.dtype}")
    B, Pk = kpm.shape
    if out is None:
        out = torch.empty(B, Pk, dtype=torch.float32, device=kpm.device)
    _require(out.dtype == torch.float32 and out.dim() == 2 and tuple(out.shape) == (B, Pk) and out.stride(1) == 1,
             f"out must be float32 [{B}, {Pk}] with contiguous rows")
    st = lib.attn_key_padding_to_additive(_ptr(kpm, "key_padding_mask"), kpm.stride(0), B, Pk, _ptr(out, "out"),
                                          out.stride(0), _stream(stream))
    _check("attn_key_padding_to_additive", st)
    return out


def attn_lse_merge(outs: Sequence[torch.Tensor], lses: Sequence[torch.Tensor], out: Optional[torch.Tensor] = None,
                   lse: Optional[torch.Tensor] = None, stream=None):
    """Merge chunk results: lse = log sum_i exp(lse_i), out = sum_i exp(lse_i - lse) out_i."""
    lib = load()
    n = len(outs)
    _require(n >= 1 and len(lses) == n, f"attn_lse_merge takes n >= 1 outputs and as many LSEs ({n}, {len(lses)})")
    if out is None:
        out = torch.empty(outs[0].shape, dtype=outs[0].dtype, device=outs[0].device)
    rows = outs[0].shape[0] * outs[0].shape[1] * outs[0].shape[2]  # B * H * P
    if lse is None:
        lse = torch.empty(lses[0].shape, dtype=torch.float32, device=outs[0].device)
    _check_f32_buffer(lse, rows, "lse")
    for i, l in enumerate(lses):
        _check_f32_buffer(l, rows, f"lses[{i}]")
    arr = (AttnTensor * n)(*[_desc(o) for o in outs])
    lptrs = (ctypes.c_void_p * n)(*[_ptr(l, f"lses[{i}]") for i, l in enumerate(lses)])
    do = _desc(out)
    st = lib.attn_lse_merge(n, arr, lptrs, ctypes.byref(do), _ptr(lse, "lse"), _stream(stream))
    _check("attn_lse_merge", st)
    return out, lse


def _cache(k_cache: torch.Tensor, v_cache: torch.Tensor) -> AttnKVCache:
    _require(k_cache.dim() == 4 and k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype,
             "K and V caches must be [num_blocks, Hkv, block_size, D] of one dtype")
    _require(k_cache.is_contiguous() and v_cache.is_contiguous(), "K and V caches must be contiguous")
    _require(_on_device(k_cache) and _on_device(v_cache), "K and V caches must be on a CUDA device")
    c = AttnKVCache()
    c.k = k_cache.data_ptr()
    c.v = v_cache.data_ptr()
    c.dtype = _dtype_code(k_cache)
    c.num_blocks = k_cache.shape[0]
    c.num_kv_heads = k_cache.shape[1]
    c.block_size = k_cache.shape[2]
    c.head_dim = k_cache.shape[3]
    return c


def kv_append(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor, pos: torch.Tensor,
              k_new: torch.Tensor, v_new: torch.Tensor, workspace: Optional[Workspace] = None, stream=None):
    """Write k_new/v_new [B, Hkv, D] at token position pos[b] of each
    sequence's paged cache (caches [num_blocks, Hkv, block_size, D])."""
    lib = load()
    _check_block_table(block_table, k_new.shape[0])
    _check_int32_vec(pos, k_new.shape[0], "pos")
    ws = workspace or _small_ws(k_cache.device)
    c = _cache(k_cache, v_cache)
    dk, dv = _desc(k_new), _desc(v_new)
    st = lib.kv_append(ctypes.byref(c), _ptr(block_table, "block_table"), block_table.stride(0),
                       block_table.shape[1], _ptr(pos, "pos"), ctypes.byref(dk), ctypes.byref(dv), ws.ptr,
                       ws.nbytes, _stream(stream))
    _check("kv_append", st)


def paged_decode_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                      ctx_lens: torch.Tensor, scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, return_lse: bool = False,
                      workspace: Optional[Workspace] = None, stream=None):
    """One query token per sequence, q [B, Hq, D], over the paged cache;
    ctx_lens int32 [B] counts the attended tokens (the appended one included)."""
    lib = load()
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_block_table(block_table, B)
    _check_int32_vec(ctx_lens, B, "ctx_lens")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, B * Hq, "lse")
    max_blocks = block_table.shape[1]
    need = paged_decode_workspace_size(B, Hq, max_blocks, k_cache.shape[2], D)
    ws = workspace
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, device=q.device)
    c = _cache(k_cache, v_cache)
    dq, do = _desc(q), _desc(out)
    st = lib.paged_decode_attn(ctypes.byref(dq), ctypes.byref(c), _ptr(block_table, "block_table"),
                               block_table.stride(0), max_blocks, _ptr(ctx_lens, "ctx_lens"), float(scale),
                               ctypes.byref(do), _ptr(lse, "lse"),
                               ws.ptr, ws.nbytes, _stream(stream))
    _check("paged_decode_attn", st)
    return (out, lse) if return_lse else out


def paged_decode_attn_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, block_table: torch.Tensor, pos: torch.Tensor,
                             scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                             lse: Optional[torch.Tensor] = None, return_lse: bool = False,
                             workspace: Optional[Workspace] = None, stream=None):
    """kv_append(pos, k_new, v_new) and the decode over tokens [0, pos[b]] in
    one launch; k_new, v_new [B, Hkv, D], pos int32 [B]."""
    lib = load()
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_block_table(block_table, B)
    _check_int32_vec(pos, B, "pos")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, B * Hq, "lse")
    max_blocks = block_table.shape[1]
    need = paged_decode_workspace_size(B, Hq, max_blocks, k_cache.shape[2], D)
    ws = workspace
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, device=q.device)
    c = _cache(k_cache, v_cache)
    dq, dk, dv, do = _desc(q), _desc(k_new), _desc(v_new), _desc(out)
    st = lib.paged_decode_attn_append(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(c),
                                      _ptr(block_table, "block_table"), block_table.stride(0), max_blocks,
                                      _ptr(pos, "pos"), float(scale), ctypes.byref(do), _ptr(lse, "lse"), ws.ptr,
                                      ws.nbytes,
                                      _stream(stream))
    _check("paged_decode_attn_append", st)
    return (out, lse) if return_lse else out


def paged_prefill_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                       start_pos: torch.Tensor, k_new: Optional[torch.Tensor] = None,
                       v_new: Optional[torch.Tensor] = None, causal: bool = True, scale: Optional[float] = None,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       return_lse: bool = False, workspace: Optional[Workspace] = None, stream=None):
    """A chunk of T tokens per sequence: q [B, Hq, T, D] at positions
    start_pos[b] + i.  With k_new / v_new ([B, Hkv, T, D]) their K/V are
    first written to the cache; queries then attend over the cache through
    the block table (causal: up to their own position)."""
    lib = load()
    B, Hq, T, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_block_table(block_table, B)
    _check_int32_vec(start_pos, B, "start_pos")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, B * Hq * T, "lse")
    ws = workspace or _small_ws(q.device)
    c = _cache(k_cache, v_cache)
    dq, do = _desc(q), _desc(out)
    dk = ctypes.byref(_desc(k_new)) if k_new is not None else None
    dv = ctypes.byref(_desc(v_new)) if v_new is not None else None
    st = lib.paged_prefill_attn(ctypes.byref(dq), dk, dv, ctypes.byref(c), _ptr(block_table, "block_table"),
                                block_table.stride(0), block_table.shape[1], _ptr(start_pos, "start_pos"),
                                int(bool(causal)), float(scale), ctypes.byref(do), _ptr(lse, "lse"), ws.ptr,
                                ws.nbytes, _stream(stream))
    _check("paged_prefill_attn", st)
    return (out, lse) if return_lse else out


def _cache_q8(kq: torch.Tensor, vq: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor) -> AttnKVCacheQ8:
    _require(kq.dtype == torch.int8 and vq.dtype == torch.int8, "INT8 caches must be int8")
    _require(kq.dim() == 4 and kq.shape == vq.shape, "INT8 caches must be [num_blocks, Hkv, block_size, D], "
             "K and V alike")
    _require(k_scale.dtype == torch.float32 and v_scale.dtype == torch.float32, "INT8 row scales must be float32")
    _require(tuple(k_scale.shape) == tuple(kq.shape[:3]) and tuple(v_scale.shape) == tuple(kq.shape[:3]),
             f"INT8 row scales must be {tuple(kq.shape[:3])}")
    for t in (kq, vq, k_scale, v_scale):
        _require(t.is_contiguous() and _on_device(t), "INT8 caches and scales must be contiguous CUDA tensors")
    c = AttnKVCacheQ8()
    c.k, c.v, c.k_scale, c.v_scale = kq.data_ptr(), vq.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr()
    c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim = kq.shape
    c.reserved = 0
    return c


def kv_append_q8(kq_cache: torch.Tensor, vq_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                 block_table: torch.Tensor, pos: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                 workspace: Optional[Workspace] = None, stream=None):
    """Quantise each sequence's new K/V rows (bf16 [B, Hkv, D]) to INT8 codes
    with one float32 scale per row and write them at pos[b]."""
    lib = load()
    _check_block_table(block_table, k_new.shape[0])
    _check_int32_vec(pos, k_new.shape[0], "pos")
    ws = workspace or _small_ws(kq_cache.device)
    c = _cache_q8(kq_cache, vq_cache, k_scale, v_scale)
    dk, dv = _desc(k_new), _desc(v_new)
    st = lib.kv_append_q8(ctypes.byref(c), _ptr(block_table, "block_table"), block_table.stride(0),
                          block_table.shape[1], _ptr(pos, "pos"), ctypes.byref(dk), ctypes.byref(dv), ws.ptr,
                          ws.nbytes, _stream(stream))
    _check("kv_append_q8", st)


def paged_decode_attn_q8(q: torch.Tensor, kq_cache: torch.Tensor, vq_cache: torch.Tensor, k_scale: torch.Tensor,
                         v_scale: torch.Tensor, block_table: torch.Tensor, ctx_lens: torch.Tensor,
                         scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                         lse: Optional[torch.Tensor] = None, return_lse: bool = False,
                         workspace: Optional[Workspace] = None, stream=None):
    """paged_decode_attn over an INT8 cache (codes int8 [N, Hkv, 16, D],
    scales float32 [N, Hkv, 16])."""
    lib = load()
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_block_table(block_table, B)
    _check_int32_vec(ctx_lens, B, "ctx_lens")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, B * Hq, "lse")
    max_blocks = block_table.shape[1]
    need = paged_decode_workspace_size(B, Hq, max_blocks, kq_cache.shape[2], D)
    ws = workspace
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, device=q.device)
    c = _cache_q8(kq_cache, vq_cache, k_scale, v_scale)
    dq, do = _desc(q), _desc(out)
    st = lib.paged_decode_attn_q8(ctypes.byref(dq), ctypes.byref(c), _ptr(block_table, "block_table"),
                                  block_table.stride(0), max_blocks, _ptr(ctx_lens, "ctx_lens"), float(scale),
                                  ctypes.byref(do), _ptr(lse, "lse"),
                                  ws.ptr, ws.nbytes, _stream(stream))
    _check("paged_decode_attn_q8", st)
    return (out, lse) if return_lse else out


def paged_decode_attn_append_q8(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, kq_cache: torch.Tensor,
                                vq_cache: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                                block_table: torch.Tensor, pos: torch.Tensor, scale: Optional[float] = None,
                                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                                return_lse: bool = False, workspace: Optional[Workspace] = None, stream=None):
    """kv_append_q8(pos, k_new, v_new) and paged_decode_attn_q8 over tokens
    [0, pos[b]] in one call; k_new, v_new bf16 [B, Hkv, D], pos int32 [B]."""
    lib = load()
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _check_block_table(block_table, B)
    _check_int32_vec(pos, B, "pos")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_f32_buffer(lse, B * Hq, "lse")
    max_blocks = block_table.shape[1]
    need = paged_decode_workspace_size(B, Hq, max_blocks, kq_cache.shape[2], D)
    ws = workspace
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, device=q.device)
    c = _cache_q8(kq_cache, vq_cache, k_scale, v_scale)
    dq, dk, dv, do = _desc(q), _desc(k_new), _desc(v_new), _desc(out)
    st = lib.paged_decode_attn_append_q8(ctypes.byref(dq), ctypes.byref(dk), ctypes.byref(dv), ctypes.byref(c),
                                         _ptr(block_table, "block_table"), block_table.stride(0), max_blocks,
                                         _ptr(pos, "pos"), float(scale), ctypes.byref(do), _ptr(lse, "lse"),
                                         ws.ptr, ws.nbytes, _stream(stream))
    _check("paged_decode_attn_append_q8", st)
    return (out, lse) if return_lse else out


def paged_kv_gather(cache: torch.Tensor, block_table: torch.Tensor, lens: torch.Tensor, max_len: int,
                    out: Optional[torch.Tensor] = None, workspace: Optional[Workspace] = None,
                    stream=None) -> torch.Tensor:
    """Contiguous copy [B, Hkv, max_len, D] of the first lens[b] tokens of each
    sequence in one paged cache tensor (K or V); rows past lens[b] untouched."""
    lib = load()
    B = lens.shape[0]
    nb, Hkv, bs, D = cache.shape
    _check_int32_vec(lens, B, "lens")
    _check_block_table(block_table, B)
    if out is None:
        out = torch.zeros((B, Hkv, max_len, D), dtype=cache.dtype, device=cache.device)
    _require(out.dtype == cache.dtype and tuple(out.shape) == (B, Hkv, max_len, D) and out.is_contiguous(),
             f"out must be contiguous {cache.dtype} [{B}, {Hkv}, {max_len}, {D}]")
    c = _cache(cache, cache)
    ws = workspace or _small_ws(cache.device)
    st = lib.paged_kv_gather(ctypes.byref(c), 0, _ptr(block_table, "block_table"), block_table.stride(0),
                             block_table.shape[1], _ptr(lens, "lens"), B, max_len, _ptr(out, "out"), ws.ptr, ws.nbytes,
                             _stream(stream))
    _check("paged_kv_gather", st)
    return out


def paged_decode_attn_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_table: torch.Tensor, ctx_lens: torch.Tensor, scale: Optional[float] = None,
                              out: torch.Tensor = None, lse: Optional[torch.Tensor] = None,
                              device_status: Optional[torch.Tensor] = None, stream=None):
    """paged_decode_attn for callers that cannot allocate device memory: the
    split-K scratch is the library's built-in 20 MiB array, so `out` (and
    `lse`, `device_status` if wanted) must be passed in.  Calls that overlap on
    the GPU race on the shared scratch."""
    lib = load()
    B, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    _require(out is not None, "the no-alloc call writes into a caller buffer: pass out")
    _check_block_table(block_table, B)
    _check_int32_vec(ctx_lens, B, "ctx_lens")
    if lse is not None:
        _check_f32_buffer(lse, B * Hq, "lse")
    if device_status is not None:
        _require(device_status.dtype in (torch.int32, torch.uint32) and device_status.numel() >= 1,
                 "device_status must be a 32-bit word")
    c = _cache(k_cache, v_cache)
    dq, do = _desc(q), _desc(out)
    st = lib.paged_decode_attn_noalloc(ctypes.byref(dq), ctypes.byref(c), _ptr(block_table, "block_table"),
                                       block_table.stride(0), block_table.shape[1], _ptr(ctx_lens, "ctx_lens"),
                                       float(scale), ctypes.byref(do), _ptr(lse, "lse"),
                                       _ptr(device_status, "device_status"),
                                       _stream(stream))
    _check("paged_decode_attn_noalloc", st)
    return out
