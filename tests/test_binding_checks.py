"""The Python binding passes raw pointers and sizes to the library, which
trusts them; so the binding checks that every buffer matches the sizes it
passes.  These tests run on the CPU with the library replaced by a recorder:
well-formed calls reach it, and a mismatched output, cache, table or scale is
rejected before any call."""
import ctypes

import pytest
import torch

import global_attention_sinks_swa_b300 as A

Hq, Hkv, D = 64, 8, 128


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append(name)
            return 0
        return fn


@pytest.fixture
def lib(monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(A, "_lib", rec)
    monkeypatch.setattr(A, "_cuda", lambda *ts: None)
    monkeypatch.setattr(A, "_stream", lambda stream=None: ctypes.c_void_p(0))
    return rec


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def _i32(*vals):
    return torch.tensor(vals, dtype=torch.int32)


def test_prefill_checks_out(lib):
    q, k, sink = _bf(1, 32, Hq, D), _bf(1, 32, Hkv, D), torch.zeros(Hq)
    A.attn_swa_sink_prefill(q, k, k, sink, out=_bf(1, 32, Hq, D))
    A.attn_ga_sink_prefill(q, k, k, sink)
    assert lib.calls == ["attn_swa_sink_prefill", "attn_ga_sink_prefill"]
    for bad in (_bf(1, 16, Hq, D), torch.zeros(1, 32, Hq, D)):
        with pytest.raises(ValueError, match="out"):
            A.attn_swa_sink_prefill(q, k, k, sink, out=bad)
    assert len(lib.calls) == 2


def test_packed_prefill_checks_out(lib):
    q, k, sink, cu = _bf(40, Hq, D), _bf(40, Hkv, D), torch.zeros(Hq), _i32(0, 15, 40)
    A.attn_swa_sink_prefill_varlen(q, k, k, cu, sink, out=_bf(40, Hq, D))
    with pytest.raises(ValueError, match="out"):
        A.attn_ga_sink_prefill_varlen(q, k, k, cu, sink, out=_bf(39, Hq, D))
    assert lib.calls == ["attn_swa_sink_prefill_varlen"]


def test_backward_checks_operands(lib):
    q, k = _bf(1, 32, Hq, D), _bf(1, 32, Hkv, D)
    lse, sink = torch.zeros(1, Hq, 32), torch.zeros(Hq)
    A.attn_sink_prefill_backward(q, k, k, q, lse, q, sink, window=128)
    with pytest.raises(ValueError, match="k"):
        A.attn_sink_prefill_backward(q, _bf(1, 32, Hkv, 64), k, q, lse, q, sink)
    with pytest.raises(ValueError, match="lse"):
        A.attn_sink_prefill_backward(q, k, k, q, lse.double(), q, sink)
    assert lib.calls == ["attn_sink_prefill_backward_workspace", "attn_sink_prefill_backward"]


def test_ring_verify_and_append_check_buffers(lib):
    B, R = 2, 131
    q, ring = _bf(8, Hq, D), _bf(B, Hkv, R, D)
    cu, sl, sink = _i32(0, 4, 8), _i32(100, 200), torch.zeros(Hq)
    A.attn_swa_sink_verify(q, cu, ring, ring, sl, sink, out=_bf(8, Hq, D))
    A.attn_swa_ring_append(_bf(8, Hkv, D), _bf(8, Hkv, D), cu, sl, ring, ring, q_max=4)
    with pytest.raises(ValueError, match="ring_v"):
        A.attn_swa_sink_verify(q, cu, ring, _bf(B, Hkv, R - 1, D), sl, sink)
    with pytest.raises(ValueError, match="out"):
        A.attn_swa_sink_verify(q, cu, ring, ring, sl, sink, out=_bf(4, Hq, D))
    with pytest.raises(ValueError, match="cu_q"):
        A.attn_swa_ring_append(_bf(8, Hkv, D), _bf(8, Hkv, D), _i32(0, 8), sl, ring, ring, q_max=4)
    assert lib.calls == ["attn_swa_sink_verify", "attn_swa_ring_append"]


def test_paged_verify_checks_pages_table_and_scales(lib):
    B, P, page = 2, 10, 64
    q, pages = _bf(8, Hq, D), _bf(P, Hkv, page, D)
    pt = torch.zeros(B, 5, dtype=torch.int32)
    cu, sl, sink = _i32(0, 4, 8), _i32(100, 300), torch.zeros(Hq)
    A.attn_ga_sink_verify(q, cu, pages, pages, pt, sl, sink, max_ctx=320, out=_bf(8, Hq, D))
    A.attn_ga_sink_verify_noalloc(q, cu, pages, pages, pt, sl, sink, max_ctx=320,
                                  out=_bf(8, Hq, D))
    A.attn_ga_paged_append(_bf(8, Hkv, D), _bf(8, Hkv, D), cu, sl, pages, pages, pt, q_max=4)
    codes = torch.zeros(P, Hkv, page, D, dtype=torch.uint8)
    ks = torch.ones(Hkv)
    A.attn_ga_sink_verify_fp8(q, cu, codes, codes, pt, sl, sink, ks, ks, max_ctx=320)
    A.attn_ga_paged_append_fp8(_bf(8, Hkv, D), _bf(8, Hkv, D), cu, sl, codes, codes, pt, ks, ks,
                               q_max=4)
    n = len(lib.calls)
    with pytest.raises(ValueError, match="v_pages"):
        A.attn_ga_sink_verify(q, cu, pages, _bf(P - 1, Hkv, page, D), pt, sl, sink, max_ctx=320)
    with pytest.raises(ValueError, match="k_pages"):
        A.attn_ga_sink_verify(q, cu, torch.zeros(P, Hkv, page, D), pages, pt, sl, sink,
                              max_ctx=320)
    with pytest.raises(ValueError, match="page_table"):
        A.attn_ga_sink_verify(q, cu, pages, pages, pt.long(), sl, sink, max_ctx=320)
    with pytest.raises(ValueError, match="seq_lens"):
        A.attn_ga_sink_verify_noalloc(q, cu, pages, pages, pt, _i32(1, 2, 3), sink, max_ctx=320,
                                      out=_bf(8, Hq, D))
    with pytest.raises(ValueError, match="k_scale"):
        A.attn_ga_sink_verify_fp8(q, cu, codes, codes, pt, sl, sink, torch.ones(Hkv - 1), ks,
                                  max_ctx=320)
    with pytest.raises(ValueError, match="v_scale"):
        A.attn_ga_paged_append_fp8(_bf(8, Hkv, D), _bf(8, Hkv, D), cu, sl, codes, codes, pt, ks,
                                   ks.double(), q_max=4)
    assert len(lib.calls) == n
