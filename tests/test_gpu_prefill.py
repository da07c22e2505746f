"""Prefill parity: the CUDA kernels (through the C ABI) against the fp64 oracle
on the same seeded inputs, element by element at small sizes (several tiles
and a ragged tail) and on sampled rows at the full 32768-token sizes."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_bf16_close, assert_f32_close

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu


def _run(kind, q, k, v, sink, window, want_lse=True):
    B, T, Hq, _ = q.shape
    lse = torch.full((B, Hq, T), float("nan"), device="cuda") if want_lse else None
    if kind == "swa":
        o = A.attn_swa_sink_prefill(q, k, v, sink, window=window, lse=lse)
    else:
        o = A.attn_ga_sink_prefill(q, k, v, sink, lse=lse)
    assert A.attn_check_device_error() == 0
    return o, lse


def _oracle(kind, q, k, v, sink, window):
    return oracle.prefill(q, k, v, sink, window if kind == "swa" else None, want_lse=True)


# ------------------------------------------------------------------ fp32 path
@pytest.mark.parametrize("kind", ["swa", "ga"])
def test_tiny_fp32_config(kind):
    """B=1, T=512, Hq=4, Hkv=1, D=64, W=128 fp32; max-abs <= 1e-4."""
    q, k, v, sink = synth.prefill_inputs(1, 512, 4, 1, 64, seed=1001, dtype=torch.float32)
    o, lse = _run(kind, q.cuda(), k.cuda(), v.cuda(), sink.cuda(), 128)
    ref, ref_lse = _oracle(kind, q, k, v, sink, 128)
    assert_f32_close(o, ref, f"fp32 {kind}")
    assert_f32_close(lse, ref_lse, f"fp32 {kind} lse")


@pytest.mark.parametrize("T,window,D", [(1, 128, 128), (77, 5, 128), (300, 128, 64), (200, 1, 64)])
def test_fp32_shapes_and_sinks(T, window, D):
    q, k, v, sink = synth.prefill_inputs(2, T, 8, 2, D, seed=T + window, dtype=torch.float32)
    sink[0], sink[3] = math.inf, -math.inf
    o, _ = _run("swa", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), window)
    ref, _ = _oracle("swa", q, k, v, sink, window)
    assert_f32_close(o, ref, "fp32 swa")


# ------------------------------------------------------------ bf16 GA tiling
@pytest.mark.parametrize("T", [1, 100, 128, 257, 640])
def test_ga_bf16_small(T):
    q, k, v, sink = synth.prefill_inputs(1, T, 8, 2, 128, seed=20 + T)
    o, lse = _run("ga", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), 0)
    ref, ref_lse = _oracle("ga", q, k, v, sink, 0)
    assert_bf16_close(o, ref, f"ga T={T}")
    assert_bf16_close(lse, ref_lse, f"ga lse T={T}")


def test_ga_bf16_batch_and_extreme_sinks():
    q, k, v, sink = synth.prefill_inputs(2, 384, 8, 1, 128, seed=77)
    sink[1], sink[2], sink[5] = math.inf, -math.inf, 30.0
    o, _ = _run("ga", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), 0)
    ref, _ = _oracle("ga", q, k, v, sink, 0)
    assert_bf16_close(o, ref, "ga sinks")
    assert torch.all(o[:, :, 1] == 0)


def test_ga_bf16_large_scores_lazy_rescale():
    """Scores with a wide dynamic range exercise the lazy running-max update."""
    q, k, v, sink = synth.prefill_inputs(1, 1024, 4, 1, 128, seed=5)
    q = (q.float() * 4).to(torch.bfloat16)
    o, _ = _run("ga", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), 0)
    ref, _ = _oracle("ga", q, k, v, sink, 0)
    assert_bf16_close(o, ref, "ga wide scores")


# ----------------------------------------------------------- bf16 SWA paths
@pytest.mark.parametrize("T,Hq,Hkv,window", [
    (16, 8, 1, 128),      # packed: one tile
    (200, 16, 2, 128),    # packed: ragged tail
    (1000, 8, 1, 128),
    (333, 8, 1, 120),     # packed, W < 128 (N = 144 still)
    (300, 8, 2, 128),     # G = 4: GA tiling with window mask
    (500, 4, 4, 50),      # G = 1: GA tiling, small window
    (130, 8, 8, 1),       # W = 1
])
def test_swa_bf16_small(T, Hq, Hkv, window):
    q, k, v, sink = synth.prefill_inputs(1, T, Hq, Hkv, 128, seed=T * 7 + window)
    o, lse = _run("swa", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), window)
    ref, ref_lse = _oracle("swa", q, k, v, sink, window)
    assert_bf16_close(o, ref, f"swa T={T} G={Hq // Hkv} W={window}")
    assert_bf16_close(lse, ref_lse, "swa lse")


@pytest.mark.parametrize("B,T,Hq,Hkv,window", [
    (2, 2500, 16, 2, 128),   # streaming runs cross (b, kv head) boundaries
    (1, 4096, 64, 8, 128),   # ~14 tiles per CTA: the 12-block K/V ring wraps repeatedly
    (1, 1500, 8, 1, 114),    # narrowest window of the streaming kernel
    (1, 1500, 8, 1, 129),    # widest window of the streaming kernel
])
def test_swa_stream_multi_tile_runs(B, T, Hq, Hkv, window):
    q, k, v, sink = synth.prefill_inputs(B, T, Hq, Hkv, 128, seed=T + window + Hkv)
    o, lse = _run("swa", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), window)
    ref, ref_lse = _oracle("swa", q, k, v, sink, window)
    assert_bf16_close(o, ref, f"swa stream B={B} T={T} Hkv={Hkv} W={window}")
    assert_bf16_close(lse, ref_lse, "swa stream lse")


def test_swa_bf16_sinks_and_batch():
    q, k, v, sink = synth.prefill_inputs(3, 150, 16, 2, 128, seed=3)
    sink[0], sink[9], sink[15] = math.inf, -math.inf, -40.0
    o, _ = _run("swa", q.cuda(), k.cuda(), v.cuda(), sink.cuda(), 128)
    ref, _ = _oracle("swa", q, k, v, sink, 128)
    assert_bf16_close(o, ref, "swa sinks")
    assert torch.all(o[:, :, 0] == 0)


def test_swa_window_ge_T_equals_ga():
    q, k, v, sink = synth.prefill_inputs(1, 100, 8, 1, 128, seed=9)
    qc, kc, vc, sc = q.cuda(), k.cuda(), v.cuda(), sink.cuda()
    o_swa, _ = _run("swa", qc, kc, vc, sc, 128)
    o_ga, _ = _run("ga", qc, kc, vc, sc, 0)
    ref, _ = _oracle("ga", q, k, v, sink, 0)
    assert_bf16_close(o_swa, ref, "swa W>=T")
    assert_bf16_close(o_ga, ref, "ga")


# ------------------------------------------------------ full-size, sampled
def _sample_rows(B, T, Hq, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = []
    for h in range(0, Hq, max(1, Hq // 8)):
        for i in list(range(0, 32)) + list(range(T - 32, T)) + list(rng.integers(0, T, n_random)):
            rows.append((int(rng.integers(0, B)), int(i), h))
    return np.array(rows, dtype=np.int32)


@pytest.mark.parametrize("kind", ["swa", "ga"])
def test_full_size_sampled_rows(kind):
    """T=32768, Hq=64, Hkv=8, D=128 (the benchmark's launch), rows sampled per head."""
    B, T, Hq, Hkv, D = 1, 32768, 64, 8, 128
    q, k, v, sink = synth.prefill_inputs(B, T, Hq, Hkv, D, seed=1002 if kind == "swa" else 1003)
    o, lse = _run(kind, q.cuda(), k.cuda(), v.cuda(), sink.cuda(), 128)
    rows = _sample_rows(B, T, Hq, 32 if kind == "ga" else 256, seed=4)
    ref, ref_lse = oracle.prefill_rows(q, k, v, sink, rows, 128 if kind == "swa" else None,
                                       want_lse=True)
    got = o[rows[:, 0], rows[:, 1], rows[:, 2]]
    got_lse = lse[rows[:, 0], rows[:, 2], rows[:, 1]]
    assert_bf16_close(got, ref, f"{kind} full-size rows")
    assert_bf16_close(got_lse, ref_lse, f"{kind} full-size lse")
    assert torch.isfinite(o).all()
