"""Packed-batch prefill parity (attn_{swa,ga}_sink_prefill_varlen): the CUDA
kernels through the C ABI against oracle.prefill_varlen on the same seeded
inputs, element by element, on batches that mix empty, one-token, ragged and
multi-tile sequences; plus the value scale, the [Hq,total] LSE layout, the
agreement with the equal-length entry points, and invalid offsets reported
through the device error word without a fault."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_bf16_close, assert_f32_close

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu


def _run(kind, q, k, v, cu, sink, window, max_seqlen=None, value_scale=1.0):
    total, Hq, _ = q.shape
    lse = torch.full((Hq, total), float("nan"), device="cuda")
    cu_d = torch.from_numpy(cu).cuda()
    if kind == "swa":
        o = A.attn_swa_sink_prefill_varlen(q, k, v, cu_d, sink, window=window,
                                           max_seqlen=max_seqlen, value_scale=value_scale, lse=lse)
    else:
        o = A.attn_ga_sink_prefill_varlen(q, k, v, cu_d, sink, max_seqlen=max_seqlen,
                                          value_scale=value_scale, lse=lse)
    assert A.attn_check_device_error() == 0
    return o, lse


MIXES = {
    "edges": [0, 1, 15, 16, 17, 0, 129, 300],
    "serving": [1000, 37, 2500, 1, 700, 16],
    "single_long": [3001],
}


@pytest.mark.parametrize("mix", list(MIXES))
def test_swa_streaming_kernel_packed(mix):
    """G = 8, W = 128: the streaming kernel (every sequence restarts the ring)."""
    lens = MIXES[mix]
    q, k, v, sink, cu = synth.packed_inputs(lens, 64, 8, 128, seed=300 + len(lens))
    sink[1], sink[2] = math.inf, -math.inf
    o, lse = _run("swa", q.cuda(), k.cuda(), v.cuda(), cu, sink.cuda(), 128)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu, sink, 128, want_lse=True)
    assert_bf16_close(o, ref, f"swa varlen {mix}")
    # head 1 has sigma = +inf: its LSE is +inf; the other heads compare as numbers
    lse = lse.cpu()
    assert bool(torch.isinf(lse[1]).all()) and bool((lse[1] > 0).all())
    keep = [h for h in range(64) if h != 1]
    assert_bf16_close(lse[keep], ref_lse[keep], f"swa varlen lse {mix}")


@pytest.mark.parametrize("window", [None, 64])
@pytest.mark.parametrize("lens", [[0, 1, 127, 128, 129, 255, 256, 257], [700, 5, 513]])
def test_ga_tiled_kernel_packed(window, lens):
    """The GA-tiled kernel: full causal, and a window it serves (64)."""
    q, k, v, sink, cu = synth.packed_inputs(lens, 16, 2, 128, seed=400 + sum(lens))
    kind = "ga" if window is None else "swa"
    o, lse = _run(kind, q.cuda(), k.cuda(), v.cuda(), cu, sink.cuda(), window or 0)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu, sink, window, want_lse=True)
    assert_bf16_close(o, ref, f"{kind} varlen {lens}")
    assert_bf16_close(lse, ref_lse, f"{kind} varlen lse {lens}")


@pytest.mark.parametrize("window", [None, 7])
def test_fp32_path_packed(window):
    lens = [0, 3, 64, 1, 200]
    q, k, v, sink, cu = synth.packed_inputs(lens, 8, 2, 64, seed=500, dtype=torch.float32)
    o, lse = _run("ga" if window is None else "swa", q.cuda(), k.cuda(), v.cuda(), cu,
                  sink.cuda(), window or 0)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu, sink, window, want_lse=True)
    assert_f32_close(o, ref, "fp32 varlen")
    assert_f32_close(lse, ref_lse, "fp32 varlen lse")


@pytest.mark.parametrize("kind,Hkv", [("swa", 8), ("ga", 8), ("swa", 2)])
def test_value_scale(kind, Hkv):
    """o = value_scale * attention (the configuration's 0.707); lse unscaled."""
    lens = [33, 290, 1]
    q, k, v, sink, cu = synth.packed_inputs(lens, 64 if Hkv == 8 else 16, Hkv, 128, seed=600)
    window = 128 if kind == "swa" else 0
    o, lse = _run(kind, q.cuda(), k.cuda(), v.cuda(), cu, sink.cuda(), window, value_scale=0.707)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu, sink, window or None, value_scale=0.707,
                                         want_lse=True)
    assert_bf16_close(o, ref, f"{kind} value_scale")
    assert_bf16_close(lse, ref_lse, f"{kind} value_scale lse")


@pytest.mark.parametrize("kind", ["swa", "ga"])
def test_equal_lengths_match_the_batched_call_bit_for_bit(kind):
    B, T = 3, 400
    q, k, v, sink = synth.prefill_inputs(B, T, 64, 8, 128, seed=700)
    q, k, v, sink = q.cuda(), k.cuda(), v.cuda(), sink.cuda()
    lse_b = torch.empty(B, 64, T, device="cuda")
    if kind == "swa":
        ob = A.attn_swa_sink_prefill(q, k, v, sink, window=128, lse=lse_b)
    else:
        ob = A.attn_ga_sink_prefill(q, k, v, sink, lse=lse_b)
    cu = np.arange(B + 1, dtype=np.int32) * T
    o, lse = _run(kind, q.reshape(B * T, 64, 128), k.reshape(B * T, 8, 128),
                  v.reshape(B * T, 8, 128), cu, sink, 128 if kind == "swa" else 0, max_seqlen=T)
    assert torch.equal(o, ob.reshape(B * T, 64, 128))
    assert torch.equal(lse, lse_b.permute(1, 0, 2).reshape(64, B * T))


@pytest.mark.parametrize("kind", ["swa", "ga"])
def test_invalid_offsets_are_reported_and_skipped(kind):
    """A decreasing span, one past total and one longer than max_seqlen set
    ATTN_DEVERR_SEQLENS; the valid sequences are still computed; the invalid
    ones' rows are left untouched."""
    lens = [40, 50, 60, 70]
    q, k, v, sink, cu = synth.packed_inputs(lens, 64, 8, 128, seed=800)
    bad = cu.copy()
    bad[2] = bad[1] - 5          # sequence 1 decreasing (and sequence 2 starts early)
    total = int(cu[-1])
    out = torch.full_like(q, 7.0).cuda()
    cu_d = torch.from_numpy(bad).cuda()
    qd, kd, vd, sd = q.cuda(), k.cuda(), v.cuda(), sink.cuda()
    A.attn_check_device_error()
    f = A.attn_swa_sink_prefill_varlen if kind == "swa" else A.attn_ga_sink_prefill_varlen
    extra = {"window": 128} if kind == "swa" else {}
    f(qd, kd, vd, cu_d, sd, max_seqlen=80, out=out, **extra)
    assert A.attn_check_device_error() & A.DEVERR_SEQLENS
    ref = oracle.prefill_varlen(q[:40], k[:40], v[:40], np.array([0, 40], np.int32), sink,
                                128 if kind == "swa" else None)
    assert_bf16_close(out[:40], ref, "valid sequence 0")
    assert bool((out[bad[1]:bad[1] + 5] == 7.0).all())  # sequence 1: untouched
    # a sequence longer than max_seqlen
    out.fill_(7.0)
    f(qd, kd, vd, torch.from_numpy(cu).cuda(), sd, max_seqlen=60, out=out, **extra)
    assert A.attn_check_device_error() & A.DEVERR_SEQLENS
    assert bool((out[cu[3]:total] == 7.0).all())
    ref3 = oracle.prefill_varlen(q[cu[2]:cu[3]], k[cu[2]:cu[3]], v[cu[2]:cu[3]],
                                 np.array([0, 60], np.int32), sink,
                                 128 if kind == "swa" else None)
    assert_bf16_close(out[cu[2]:cu[3]], ref3, "valid sequence 2")
    assert A.attn_check_device_error() == 0


def test_host_rejects_bad_arguments():
    q = torch.zeros(10, 64, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(10, 8, 128, dtype=torch.bfloat16, device="cuda")
    sink = torch.zeros(64, device="cuda")
    cu = torch.tensor([0, 10], dtype=torch.int32, device="cuda")
    with pytest.raises(A.AttnError) as e:
        A.attn_swa_sink_prefill_varlen(q, k, k, cu, sink, window=0, max_seqlen=10)
    assert e.value.status == A.ATTN_ERR_INVALID_ARG
    with pytest.raises(A.AttnError) as e:
        A.attn_ga_sink_prefill_varlen(q, k, k, cu, sink, max_seqlen=10, value_scale=math.inf)
    assert e.value.status == A.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", ["swa", "ga"])
def test_many_sequences(kind):
    """100 sequences (zeros among them): the streaming kernel locates each CTA's
    first tile with a warp scan over chunks of 32 sequences."""
    lens = synth.packed_lengths(100, 1, 300, 1234)
    lens[::7] = 0
    lens[3] = 17
    q, k, v, sink, cu = synth.packed_inputs(lens, 64 if kind == "swa" else 16,
                                            8 if kind == "swa" else 2, 128, seed=1235)
    o, lse = _run(kind, q.cuda(), k.cuda(), v.cuda(), cu, sink.cuda(), 128 if kind == "swa" else 0)
    ref, ref_lse = oracle.prefill_varlen(q, k, v, cu, sink, 128 if kind == "swa" else None,
                                         want_lse=True)
    assert_bf16_close(o, ref, f"{kind} 100 sequences")
    assert_bf16_close(lse, ref_lse, f"{kind} 100 sequences lse")
