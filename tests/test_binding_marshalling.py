"""Every binding function, marshalled all the way to its C call, on the CPU.

The library is replaced by a recorder that converts each argument with the
ctypes type the real entry point declares (the binding's own signature
table), so a misspelt argument, a wrong count or a value ctypes cannot pass
fails here rather than on a GPU machine.  The tensors are CPU tensors; the
binding's device predicate is patched to accept them.  Nothing is computed:
the recorder returns ATTN_OK (or a size) without touching any buffer."""
import ctypes

import pytest
import torch

import masked_attention_paged_gb300 as lib


class _Recorder:
    def __init__(self):
        self.sig = lib._signatures()
        self.calls = []

    def __getattr__(self, name):
        if name not in self.sig:
            raise AttributeError(name)
        res, argtypes = self.sig[name]

        def call(*args):
            assert len(args) == len(argtypes), f"{name}: {len(args)} arguments, the C entry point takes {len(argtypes)}"
            for i, (a, t) in enumerate(zip(args, argtypes)):
                try:
                    t.from_param(a)
                except TypeError as e:
                    raise AssertionError(f"{name}: argument {i} ({a!r}) does not convert to {t}: {e}") from e
            self.calls.append(name)
            return 4096 if res is ctypes.c_size_t else 0

        return call


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(lib, "load", lambda build_if_missing=False: r)
    monkeypatch.setattr(lib, "_on_device", lambda t: True)
    monkeypatch.setattr(lib, "_default_ws", {})  # the CPU workspaces made here stay here
    return r


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def test_attention_calls(rec):
    q = _bf(2, 4, 8, 64)
    mask = torch.zeros(2, 8)
    o, l = lib.attn_fwd(q, q, q, mask, stream=0)
    assert o.shape == q.shape and l.shape == (2, 4, 8)
    lib.attn_fwd(q, q, q, None, 0.1, return_lse=False, workspace=lib.Workspace(256, device="cpu"), stream=0)
    lib.attn_fwd_varlen(q, q, q, torch.full((2,), 5, dtype=torch.int32), stream=0)
    lib.key_padding_to_additive(torch.zeros(2, 8, dtype=torch.bool), stream=0)
    lib.attn_lse_merge([q, q], [l, l.clone()], stream=0)
    assert rec.calls == ["attn_fwd_workspace_size_for", "attn_fwd", "attn_fwd", "attn_fwd_workspace_size_for",
                         "attn_fwd_varlen", "attn_key_padding_to_additive", "attn_lse_merge"]


def test_paged_calls(rec):
    B, Hq, Hkv, D, nb, mb = 3, 8, 2, 128, 10, 4
    q = _bf(B, Hq, D)
    kc = _bf(nb, Hkv, 16, D)
    bt = torch.zeros(B, mb, dtype=torch.int32)
    lens = torch.ones(B, dtype=torch.int32)
    kn = _bf(B, Hkv, D)
    lib.kv_append(kc, kc, bt, lens, kn, kn, stream=0)
    lib.paged_decode_attn(q, kc, kc, bt, lens, return_lse=True, stream=0)
    lib.paged_decode_attn_append(q, kn, kn, kc, kc, bt, lens, return_lse=True, stream=0)
    qp = _bf(B, Hq, 5, D)
    lib.paged_prefill_attn(qp, kc, kc, bt, lens, k_new=_bf(B, Hkv, 5, D), v_new=_bf(B, Hkv, 5, D),
                           return_lse=True, stream=0)
    lib.paged_prefill_attn(qp, kc, kc, bt, lens, causal=False, stream=0)
    lib.paged_kv_gather(kc, bt, lens, 20, stream=0)
    lib.paged_decode_attn_noalloc(q, kc, kc, bt, lens, out=torch.empty_like(q), lse=torch.empty(B, Hq),
                                  device_status=torch.zeros(1, dtype=torch.int32), stream=0)
    kq = torch.zeros(nb, Hkv, 16, D, dtype=torch.int8)
    sc = torch.zeros(nb, Hkv, 16)
    lib.kv_append_q8(kq, kq, sc, sc, bt, lens, kn, kn, stream=0)
    lib.paged_decode_attn_q8(q, kq, kq, sc, sc, bt, lens, return_lse=True, stream=0)
    lib.paged_decode_attn_append_q8(q, kn, kn, kq, kq, sc, sc, bt, lens, return_lse=True, stream=0)
    assert [c for c in rec.calls if c != "paged_decode_workspace_size"] == [
        "kv_append", "paged_decode_attn", "paged_decode_attn_append", "paged_prefill_attn", "paged_prefill_attn",
        "paged_kv_gather", "paged_decode_attn_noalloc", "kv_append_q8", "paged_decode_attn_q8",
        "paged_decode_attn_append_q8"]


def test_workspace_and_status_calls(rec):
    ws = lib.Workspace(100, device="cpu")
    assert ws.nbytes == 256
    assert ws.status(stream=0) == 0
    ws.reset(stream=0)
    assert lib.attn_fwd_workspace_size() == 4096
    assert lib.paged_decode_workspace_size(4, 8, 10) == 4096
    assert rec.calls == ["attn_check_device_status", "attn_reset_device_status", "attn_fwd_workspace_size",
                         "paged_decode_workspace_size"]


def test_signature_table_covers_the_exported_symbols():
    assert set(lib.exported_symbols()) <= set(lib._signatures())
