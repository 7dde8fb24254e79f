"""The C-ABI boundary without a GPU: the library loads, exports every function
include/libattn.h declares, sizes workspaces as documented, and rejects bad
arguments on the host before anything is launched.

Every call below carries exactly one bad argument, so validation returns
before the library touches the CUDA runtime; the fake device addresses are
never dereferenced."""
import ctypes
import os
import re
import subprocess

import pytest

import masked_attention_paged_gb300 as lib
from masked_attention_paged_gb300 import AttnKVCache, AttnTensor

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "libattn.h")
FAKE = 0x7f0000010000  # 64 KiB aligned, never dereferenced

OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT, BOUNDS, WORKSPACE = range(7)


@pytest.fixture(scope="module")
def L():
    return lib.load(build_if_missing=True)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for f in ["attn_fwd", "attn_lse_merge", "kv_append", "paged_decode_attn"]:
        assert f in names


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(L, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib.library_path()], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in names:
        assert name in exported, name


def test_status_strings_and_version(L):
    assert L.attn_version() >= 100
    assert L.attn_status_string(OK) == b"ATTN_OK"
    assert L.attn_status_string(BOUNDS) == b"ATTN_ERR_DEVICE_BOUNDS"
    assert L.attn_status_string(99) == b"ATTN_UNKNOWN_STATUS"


def test_workspace_sizes(L):
    assert L.attn_fwd_workspace_size() == 256
    # with the per-tile key bounds: one float per (batch, KV head, 128-key tile), D = 64 only
    assert L.attn_fwd_workspace_size_for(1, 16, 32000, 64) == 256 + (16 * 250 * 4 + 255) // 256 * 256
    assert L.attn_fwd_workspace_size_for(2, 4, 129, 64) == 256 + 256
    assert L.attn_fwd_workspace_size_for(1, 24, 16380, 128) == 256
    assert L.attn_fwd_workspace_size_for(1, 16, -1, 64) == 0
    assert L.kv_append_workspace_size() == 256
    # decode: status block + partials [B, Hq, n_split, D] + lse [B, Hq, n_split], split = 1024 tokens,
    # then 8-byte split counts (B * Hq of them bound the B * Hkv used) at an 8-byte boundary
    n_split = -(-513 * 16 // 1024)
    assert n_split == 9
    part = 64 * 32 * n_split * (128 + 1) * 4
    part = (part + 7) // 8 * 8 + 64 * 32 * 8
    assert L.paged_decode_workspace_size(64, 32, 513, 16, 128) == 256 + (part + 255) // 256 * 256
    # linear in the longest context, never quadratic
    a, b, c = (L.paged_decode_workspace_size(8, 32, m, 16, 128) for m in (1024, 2048, 3072))
    assert abs((c - b) - (b - a)) <= 256 and c > b > a


def _t(shape, dtype=1, stride=None, data=FAKE):
    t = AttnTensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    if stride is None:
        stride, acc = [], 1
        for s in reversed(shape):
            stride.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, stride)):
        t.shape[i] = s
        t.stride[i] = st
    return t


def _fwd(L, q, k, v, out, ws=FAKE, ws_bytes=256, mask=None, mstride=0, scale=0.125):
    return L.attn_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), mask, mstride, scale, ctypes.byref(out),
                      None, ws, ws_bytes, None)


GOOD = dict(q=(1, 4, 100, 64), k=(1, 2, 90, 64))


@pytest.mark.parametrize("case,expect", [
    ("q_ndim", INVALID), ("head_dim_mismatch", INVALID), ("gqa_not_divisible", INVALID),
    ("dtype_mismatch", INVALID), ("inner_stride", INVALID), ("out_shape", INVALID),
    ("no_workspace", WORKSPACE), ("small_workspace", WORKSPACE), ("misaligned_workspace", WORKSPACE),
    ("bf16_d96", UNSUPPORTED), ("f32_d130", UNSUPPORTED), ("misaligned_q", INVALID),
    ("odd_row_stride", INVALID), ("nan_scale", INVALID), ("mask_stride", INVALID), ("null_data", INVALID),
])
def test_attn_fwd_rejects(L, case, expect):
    q, k = list(GOOD["q"]), list(GOOD["k"])
    dt = 1
    kw = {}
    if case == "q_ndim":
        qt = _t(q[1:])
    else:
        qt = _t(q)
    kt, vt, ot = _t(k), _t(k), _t(q)
    if case == "head_dim_mismatch":
        kt = _t(k[:3] + [128]); vt = _t(k[:3] + [128])
    elif case == "gqa_not_divisible":
        kt = _t([1, 3, 90, 64]); vt = _t([1, 3, 90, 64])
    elif case == "dtype_mismatch":
        kt = _t(k, dtype=0)
    elif case == "inner_stride":
        qt = _t(q, stride=[4 * 100 * 128, 100 * 128, 128, 2])
    elif case == "out_shape":
        ot = _t([1, 4, 99, 64])
    elif case == "no_workspace":
        kw = dict(ws=None)
    elif case == "small_workspace":
        kw = dict(ws_bytes=128)
    elif case == "misaligned_workspace":
        kw = dict(ws=FAKE + 16)
    elif case == "bf16_d96":
        qt, kt, vt, ot = _t([1, 4, 100, 96]), _t([1, 2, 90, 96]), _t([1, 2, 90, 96]), _t([1, 4, 100, 96])
    elif case == "f32_d130":
        qt, kt, vt, ot = (_t([1, 4, 100, 132], 0), _t([1, 2, 90, 132], 0), _t([1, 2, 90, 132], 0),
                          _t([1, 4, 100, 132], 0))
    elif case == "misaligned_q":
        qt = _t(q, data=FAKE + 2)
    elif case == "odd_row_stride":
        qt = _t(q, stride=[4 * 100 * 68, 100 * 68, 68 - 1, 1])
    elif case == "nan_scale":
        kw = dict(scale=float("nan"))
    elif case == "mask_stride":
        qt, ot = _t([2, 4, 100, 64]), _t([2, 4, 100, 64])
        kt, vt = _t([2, 2, 90, 64]), _t([2, 2, 90, 64])
        kw = dict(mask=FAKE, mstride=89)
    elif case == "null_data":
        vt = _t(k, data=0)
    assert _fwd(L, qt, kt, vt, ot, **kw) == expect


def test_attn_fwd_empty_is_a_no_op(L):
    # zero query rows: validated, nothing launched
    assert _fwd(L, _t([1, 4, 0, 64]), _t([1, 2, 90, 64]), _t([1, 2, 90, 64]), _t([1, 4, 0, 64])) == OK
    assert _fwd(L, _t([0, 4, 10, 64]), _t([0, 2, 90, 64]), _t([0, 2, 90, 64]), _t([0, 4, 10, 64])) == OK


def _merge(L, outs, lses, out, n=None):
    arr = (AttnTensor * len(outs))(*outs)
    lp = (ctypes.c_void_p * len(lses))(*lses)
    return L.attn_lse_merge(len(outs) if n is None else n, arr, lp, ctypes.byref(out), None, None)


def test_lse_merge_rejects(L):
    o = _t([1, 2, 10, 128])
    assert _merge(L, [o, o], [FAKE, FAKE], o, n=0) == INVALID
    assert _merge(L, [o] * 9, [FAKE] * 9, o) == INVALID
    assert _merge(L, [o, _t([1, 2, 11, 128])], [FAKE, FAKE], o) == INVALID
    assert _merge(L, [o, _t([1, 2, 10, 128], 0)], [FAKE, FAKE], o) == INVALID
    assert _merge(L, [o, o], [FAKE, 0], o) == INVALID
    o12 = _t([1, 2, 10, 12])
    assert _merge(L, [o12, o12], [FAKE, FAKE], o12) == UNSUPPORTED


def _cache(bs=16, D=128, dtype=1, nb=100, H=8):
    c = AttnKVCache()
    c.k, c.v, c.dtype, c.block_size, c.num_blocks, c.num_kv_heads, c.head_dim = FAKE, FAKE, dtype, bs, nb, H, D
    return c


def test_kv_append_rejects(L):
    kn = _t([4, 8, 128])
    def call(c=None, bt=FAKE, pos=FAKE, k=kn, v=kn, ws=FAKE, mb=10, bts=10):
        c = c or _cache()
        return L.kv_append(ctypes.byref(c), bt, bts, mb, pos, ctypes.byref(k), ctypes.byref(v), ws, 256, None)
    assert call(c=_cache(bs=32)) == UNSUPPORTED
    assert call(c=_cache(dtype=0)) == UNSUPPORTED
    assert call(c=_cache(D=96)) == UNSUPPORTED
    assert call(pos=None) == INVALID
    assert call(bt=None) == INVALID
    assert call(k=_t([4, 4, 128])) == INVALID
    assert call(v=_t([4, 8, 128], 0)) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(mb=0) == INVALID
    assert call(bts=5) == INVALID


def test_paged_decode_rejects(L):
    need = L.paged_decode_workspace_size(4, 32, 10, 16, 128)
    def call(q=None, c=None, bt=FAKE, lens=FAKE, ws_bytes=need, mb=10, out=None, scale=0.1):
        q = q or _t([4, 32, 128])
        out = out or _t([4, 32, 128])
        c = c or _cache()
        return L.paged_decode_attn(ctypes.byref(q), ctypes.byref(c), bt, 10, mb, lens, scale, ctypes.byref(out),
                                   None, FAKE, ws_bytes, None)
    assert call(q=_t([4, 12, 128]), out=_t([4, 12, 128]), c=_cache(H=4)) == UNSUPPORTED  # group of 3
    assert call(q=_t([4, 30, 128]), out=_t([4, 30, 128])) == INVALID  # 30 % 8
    assert call(q=_t([4, 32, 64]), out=_t([4, 32, 64])) == INVALID  # D differs from the cache
    assert call(ws_bytes=need - 256) == WORKSPACE
    assert call(lens=None) == INVALID
    assert call(mb=0) == INVALID
    assert call(q=_t([4, 32, 128], 0)) == UNSUPPORTED
    assert call(scale=float("inf")) == INVALID


def test_attn_fwd_varlen_rejects(L):
    q, k = _t(list(GOOD["q"])), _t(list(GOOD["k"]))
    def call(kl=FAKE, ws=FAKE, qq=q):
        return L.attn_fwd_varlen(ctypes.byref(qq), ctypes.byref(k), ctypes.byref(k), kl, 0.125, ctypes.byref(qq),
                                 None, ws, 256, None)
    assert call(kl=None) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(qq=_t([1, 4, 100, 128])) == INVALID  # head dim differs from k
    assert call(qq=_t([1, 4, 0, 64])) == OK  # zero query rows: nothing launched


def test_key_padding_converter_rejects(L):
    def call(kpm=FAKE, ks=300, b=3, n=300, out=FAKE, os_=300):
        return L.attn_key_padding_to_additive(kpm, ks, b, n, out, os_, None)
    assert call(b=-1) == INVALID
    assert call(n=-1) == INVALID
    assert call(kpm=None) == INVALID
    assert call(out=None) == INVALID
    assert call(ks=299) == INVALID
    assert call(os_=299) == INVALID
    assert call(out=FAKE + 2) == INVALID  # float output must be 4-byte aligned
    assert call(b=0) == OK and call(n=0) == OK


def test_fused_decode_rejects(L):
    need = L.paged_decode_workspace_size(4, 32, 10, 16, 128)
    kn = _t([4, 8, 128])
    def call(k=kn, v=kn, ws_bytes=need):
        q, out, c = _t([4, 32, 128]), _t([4, 32, 128]), _cache()
        return L.paged_decode_attn_append(ctypes.byref(q), None if k is None else ctypes.byref(k),
                                          None if v is None else ctypes.byref(v), ctypes.byref(c), FAKE, 10, 10,
                                          FAKE, 0.1, ctypes.byref(out), None, FAKE, ws_bytes, None)
    assert call(k=None) == INVALID
    assert call(v=None) == INVALID
    assert call(k=_t([4, 4, 128])) == INVALID  # heads differ from the cache
    assert call(v=_t([4, 8, 128], 0)) == INVALID  # f32
    assert call(k=_t([3, 8, 128]), v=_t([3, 8, 128])) == INVALID  # batch differs from q
    assert call(ws_bytes=need - 256) == WORKSPACE


def test_paged_prefill_rejects(L):
    def call(q=None, k=None, v=None, c=None, sp=FAKE, causal=1, out=None, ws=FAKE, scale=0.1, bts=10):
        q = q or _t([2, 8, 40, 128])
        out = out or _t([2, 8, 40, 128])
        c = c or _cache()
        return L.paged_prefill_attn(ctypes.byref(q), None if k is None else ctypes.byref(k),
                                    None if v is None else ctypes.byref(v), ctypes.byref(c), FAKE, bts, 10, sp,
                                    causal, scale, ctypes.byref(out), None, ws, 256, None)
    kn = _t([2, 8, 40, 128])
    assert call(k=kn) == INVALID  # k_new without v_new
    assert call(k=_t([2, 8, 39, 128]), v=_t([2, 8, 39, 128])) == INVALID  # chunk length differs from q
    assert call(k=_t([2, 4, 40, 128]), v=_t([2, 4, 40, 128])) == INVALID  # heads differ from the cache
    assert call(q=_t([2, 8, 40, 128], 0), out=_t([2, 8, 40, 128], 0)) == UNSUPPORTED  # f32 queries
    assert call(q=_t([2, 8, 40, 64]), out=_t([2, 8, 40, 64])) == INVALID  # D differs from the cache
    assert call(q=_t([2, 12, 40, 128]), out=_t([2, 12, 40, 128])) == INVALID  # 12 % 8
    assert call(causal=2) == INVALID
    assert call(sp=None) == INVALID
    assert call(ws=None) == WORKSPACE
    assert call(scale=float("nan")) == INVALID
    assert call(bts=5) == INVALID
    assert call(q=_t([2, 8, 0, 128]), out=_t([2, 8, 0, 128])) == OK  # empty chunk: nothing launched


def _cache_q8(D=128, nb=100, H=8, bs=16, k=FAKE, ks=FAKE):
    c = lib.AttnKVCacheQ8()
    c.k, c.v, c.k_scale, c.v_scale = k, FAKE, ks, FAKE
    c.num_blocks, c.block_size, c.num_kv_heads, c.head_dim, c.reserved = nb, bs, H, D, 0
    return c


def test_q8_calls_reject(L):
    kn = _t([4, 8, 128])
    def app(c=None, k=kn):
        c = c or _cache_q8()
        return L.kv_append_q8(ctypes.byref(c), FAKE, 10, 10, FAKE, ctypes.byref(k), ctypes.byref(kn), FAKE, 256, None)
    assert app(c=_cache_q8(ks=None)) == INVALID
    assert app(c=_cache_q8(ks=FAKE + 4)) == INVALID  # scales must be 16-byte aligned
    assert app(c=_cache_q8(bs=32)) == UNSUPPORTED
    assert app(c=_cache_q8(D=96)) == UNSUPPORTED
    assert app(k=_t([4, 8, 64])) == INVALID  # head dim differs from the cache
    need = L.paged_decode_workspace_size(4, 32, 10, 16, 128)
    def dec(c=None, ws_bytes=need, q=None):
        c = c or _cache_q8()
        q = q or _t([4, 32, 128])
        out = _t([4, 32, 128])
        return L.paged_decode_attn_q8(ctypes.byref(q), ctypes.byref(c), FAKE, 10, 10, FAKE, 0.1, ctypes.byref(out),
                                      None, FAKE, ws_bytes, None)
    assert dec(c=_cache_q8(k=None)) == INVALID
    assert dec(ws_bytes=need - 256) == WORKSPACE
    assert dec(q=_t([4, 32, 128], 0)) == UNSUPPORTED  # f32 queries
    def fused(k=kn, v=kn, c=None, ws_bytes=need):
        c = c or _cache_q8()
        q, out = _t([4, 32, 128]), _t([4, 32, 128])
        return L.paged_decode_attn_append_q8(ctypes.byref(q), None if k is None else ctypes.byref(k),
                                             None if v is None else ctypes.byref(v), ctypes.byref(c), FAKE, 10, 10,
                                             FAKE, 0.1, ctypes.byref(out), None, FAKE, ws_bytes, None)
    assert fused(k=None) == INVALID
    assert fused(v=None) == INVALID
    assert fused(k=_t([4, 8, 64])) == INVALID  # head dim differs from the cache
    assert fused(k=_t([3, 8, 128])) == INVALID  # batch differs from q
    assert fused(c=_cache_q8(ks=None)) == INVALID
    assert fused(ws_bytes=need - 256) == WORKSPACE
