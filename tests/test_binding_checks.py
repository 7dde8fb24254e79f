"""The binding's checks on arguments that reach libattn as bare pointers.

LSE buffers, masks, block tables and per-sequence positions or lengths carry
no shape the C side could check, so the binding checks their dtype, size and
layout before any call.  These run without a GPU: every case is rejected
before the library is called (the tensors are on the CPU, and a check that
passed would stop at the device check instead)."""
import pytest
import torch

import masked_attention_paged_gb300 as lib


@pytest.fixture(autouse=True)
def _library():
    lib.load()


def _q(B=2, H=4, P=8, D=64):
    return torch.zeros(B, H, P, D, dtype=torch.bfloat16)


def test_attn_fwd_rejects_a_short_or_mistyped_lse():
    q = k = v = _q()
    with pytest.raises(ValueError, match="lse must hold 64 elements"):
        lib.attn_fwd(q, k, v, lse=torch.zeros(2, 4, 7))
    with pytest.raises(ValueError, match="lse must be float32"):
        lib.attn_fwd(q, k, v, lse=torch.zeros(2, 4, 8, dtype=torch.float64))
    with pytest.raises(ValueError, match="lse must be contiguous"):
        lib.attn_fwd(q, k, v, lse=torch.zeros(2, 8, 4).transpose(1, 2))


def test_attn_fwd_rejects_a_mask_of_the_wrong_shape_or_kind():
    q = k = v = _q()
    lse = torch.zeros(2, 4, 8)
    with pytest.raises(ValueError, match="key_pad_mask must be float32"):
        lib.attn_fwd(q, k, v, torch.zeros(2, 8, dtype=torch.bool), lse=lse)
    with pytest.raises(ValueError, match=r"key_pad_mask must be \[2, 8\]"):
        lib.attn_fwd(q, k, v, torch.zeros(1, 8), lse=lse)
    with pytest.raises(ValueError, match=r"key_pad_mask must be \[2, 8\]"):
        lib.attn_fwd(q, k, v, torch.zeros(2, 7), lse=lse)
    # the shapes right, only the device left to object
    with pytest.raises(ValueError, match="key_pad_mask must be on a CUDA device"):
        lib.attn_fwd(q, k, v, torch.zeros(2, 8), lse=lse)


def test_attn_fwd_varlen_rejects_lengths_that_are_not_int32_per_row():
    q = k = v = _q()
    with pytest.raises(ValueError, match="key_lens must be int32"):
        lib.attn_fwd_varlen(q, k, v, torch.zeros(2, dtype=torch.int64))
    with pytest.raises(ValueError, match=r"key_lens must be contiguous \[2\]"):
        lib.attn_fwd_varlen(q, k, v, torch.zeros(3, dtype=torch.int32))


def test_merge_rejects_mismatched_partials():
    o = _q()
    l = torch.zeros(2, 4, 8)
    with pytest.raises(ValueError, match="as many LSEs"):
        lib.attn_lse_merge([o, o], [l])
    with pytest.raises(ValueError, match=r"lses\[1\] must hold 64 elements"):
        lib.attn_lse_merge([o, o], [l, torch.zeros(2, 4, 4)])
    with pytest.raises(ValueError, match=r"lse must hold 64 elements"):
        lib.attn_lse_merge([o, o], [l, l], lse=torch.zeros(10))


def _decode_args(B=3, Hq=8, Hkv=2, D=128, nb=10, mb=4):
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16)
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.bfloat16)
    bt = torch.zeros(B, mb, dtype=torch.int32)
    lens = torch.ones(B, dtype=torch.int32)
    return q, kc, bt, lens


def test_decode_rejects_bad_tables_and_lengths():
    q, kc, bt, lens = _decode_args()
    with pytest.raises(ValueError, match="block_table must be int32"):
        lib.paged_decode_attn(q, kc, kc, bt.long(), lens)
    with pytest.raises(ValueError, match=r"block_table must be \[>= 3, max_blocks\]"):
        lib.paged_decode_attn(q, kc, kc, bt[:2], lens)
    with pytest.raises(ValueError, match=r"block_table must be \[>= 3, max_blocks\]"):
        lib.paged_decode_attn(q, kc, kc, bt.t(), lens)
    with pytest.raises(ValueError, match=r"ctx_lens must be contiguous \[3\]"):
        lib.paged_decode_attn(q, kc, kc, bt, lens[:2])
    with pytest.raises(ValueError, match="lse must hold 24 elements"):
        lib.paged_decode_attn(q, kc, kc, bt, lens, lse=torch.zeros(3, 4))


def test_append_and_prefill_reject_bad_positions():
    q, kc, bt, lens = _decode_args()
    kn = torch.zeros(3, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="pos must be int32"):
        lib.kv_append(kc, kc, bt, lens.long(), kn, kn)
    with pytest.raises(ValueError, match=r"pos must be contiguous \[3\]"):
        lib.kv_append(kc, kc, bt, torch.zeros(3, 2, dtype=torch.int32), kn, kn)
    qp = torch.zeros(3, 8, 5, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"start_pos must be contiguous \[3\]"):
        lib.paged_prefill_attn(qp, kc, kc, bt, torch.zeros(4, dtype=torch.int32))


def test_gather_output_must_fit():
    q, kc, bt, lens = _decode_args()
    with pytest.raises(ValueError, match=r"out must be contiguous torch.bfloat16 \[3, 2, 40, 128\]"):
        lib.paged_kv_gather(kc, bt, lens, 40, out=torch.zeros(3, 2, 39, 128, dtype=torch.bfloat16))


def test_caches_must_match_and_int8_scales_must_fit():
    q, kc, bt, lens = _decode_args()
    with pytest.raises(ValueError, match="K and V caches must be"):
        lib.paged_decode_attn(q, kc, kc[:5], bt, lens)
    kq = torch.zeros(10, 2, 16, 128, dtype=torch.int8)
    sc = torch.zeros(10, 2, 16)
    with pytest.raises(ValueError, match="INT8 row scales must be"):
        lib.paged_decode_attn_q8(q, kq, kq, sc, sc[:, :, :8], bt, lens)
    with pytest.raises(ValueError, match="INT8 caches must be int8"):
        lib.paged_decode_attn_q8(q, kq.to(torch.uint8), kq, sc, sc, bt, lens)
