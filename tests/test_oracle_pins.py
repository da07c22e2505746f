"""Pins of the fp64 oracle against things other than itself.

Each test compares the C oracle with an independent formulation or a fact that
the mathematics fixes: the numpy brute force (full matrix + sink column +
library softmax), torch's own scaled-dot-product attention in fp64 (a library
routine; with GQA it fixes the head map h -> h // (Hq/Hkv)), and closed forms
and invariants of softmax with a sink column (sink = -inf reduces to plain
softmax, sink = +inf gives zero output, row weights sum to 1 - p_sink,
W = 1 gives o_i = v_i (1 - p_sink), W >= T equals global attention, equal keys
give a uniform average).  CPU only.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import brute

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(B, T, Hq, Hkv, D, seed, sink_override=None):
    q, k, v, sink = synth.prefill_inputs(B, T, Hq, Hkv, D, seed, dtype=torch.float32)
    if sink_override is not None:
        sink = torch.tensor(sink_override, dtype=torch.float32)
    return q, k, v, sink


CASES = [
    # B, T, Hq, Hkv, D, window, sinks
    (1, 1, 2, 1, 8, None, None),
    (1, 5, 4, 1, 8, 3, None),
    (2, 17, 4, 2, 16, 4, None),
    (1, 33, 8, 2, 8, 1, None),
    (1, 64, 4, 4, 16, 16, None),
    (2, 40, 6, 3, 8, 100, None),
    (1, 29, 4, 2, 8, 7, [-math.inf, math.inf, 0.5, -2.0]),
    (1, 48, 4, 1, 16, None, [3.0, -math.inf, math.inf, -0.25]),
]


@pytest.mark.parametrize("B,T,Hq,Hkv,D,window,sinks", CASES)
def test_c_oracle_equals_brute_force(B, T, Hq, Hkv, D, window, sinks):
    q, k, v, sink = _inputs(B, T, Hq, Hkv, D, seed=11 + T, sink_override=sinks)
    scale = 1.0 / math.sqrt(D)
    o, lse, ps = oracle.prefill(q, k, v, sink, window, scale, want_lse=True, want_psink=True)
    ob, psb, lseb = brute.prefill(q.numpy(), k.numpy(), v.numpy(), sink.numpy(), window, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ps, psb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv", [(4, 1), (4, 2), (8, 8), (8, 2)])
def test_no_sink_full_window_equals_torch_causal_sdpa(Hq, Hkv):
    """sink = -inf and W >= T: plain causal softmax attention (library routine)."""
    B, T, D = 2, 37, 16
    q, k, v, _ = _inputs(B, T, Hq, Hkv, D, seed=5)
    sink = torch.full((Hq,), -math.inf)
    scale = 0.3
    for window in (None, T, T + 50):
        o = oracle.prefill(q, k, v, sink, window, scale)
        ref = F.scaled_dot_product_attention(
            q.double().transpose(1, 2), k.double().transpose(1, 2), v.double().transpose(1, 2),
            is_causal=True, scale=scale, enable_gqa=True).transpose(1, 2)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("window", [1, 2, 9, 128])
def test_sink_as_extra_key_column_equals_torch_sdpa(window):
    """The sink as an extra key whose score is sigma_h and whose value is zero,
    through torch's scaled-dot-product attention with an additive mask."""
    B, T, Hq, Hkv, D = 1, 150, 8, 2, 16
    q, k, v, sink = _inputs(B, T, Hq, Hkv, D, seed=7)
    scale = 1.0 / math.sqrt(D)
    o = oracle.prefill(q, k, v, sink, window, scale)
    qd, kd, vd = (x.double().transpose(1, 2) for x in (q, k, v))          # [B,H,T,D]
    kd = torch.cat([kd, torch.zeros(B, Hkv, 1, D, dtype=torch.float64)], dim=2)
    vd = torch.cat([vd, torch.zeros(B, Hkv, 1, D, dtype=torch.float64)], dim=2)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    allowed = (j <= i) & (j > i - window)
    bias = torch.where(allowed, 0.0, -math.inf).double()                  # [T,T]
    bias = bias[None].expand(Hq, T, T)
    sink_col = sink.double()[:, None, None].expand(Hq, T, 1)
    bias = torch.cat([bias, sink_col], dim=2)[None]                        # [1,Hq,T,T+1]
    ref = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=bias, scale=scale,
                                         enable_gqa=True).transpose(1, 2)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_sink_plus_inf_gives_zero_output():
    q, k, v, _ = _inputs(1, 20, 4, 2, 8, seed=3)
    sink = torch.tensor([math.inf, 0.0, math.inf, -1.0])
    o, lse, ps = oracle.prefill(q, k, v, sink, 5, 0.5, want_lse=True, want_psink=True)
    assert np.all(o[:, :, [0, 2]] == 0.0)
    assert np.all(ps[:, [0, 2]] == 1.0) and np.all(np.isposinf(lse[:, [0, 2]]))
    assert np.all(np.abs(o[:, :, [1, 3]]).sum(-1) > 0)


@pytest.mark.parametrize("window", [None, 1, 6])
def test_row_weights_sum_to_one_minus_psink(window):
    """With every value vector equal to ones, each output element is the sum
    of the row's attention weights, which must be 1 - p_sink."""
    B, T, Hq, Hkv, D = 1, 30, 4, 2, 8
    q, k, _, sink = _inputs(B, T, Hq, Hkv, D, seed=9)
    v = torch.ones(B, T, Hkv, D)
    o, ps = oracle.prefill(q, k, v, sink, window, 0.4, want_psink=True)
    expect = (1.0 - ps).transpose(0, 2, 1)[..., None]                      # [B,T,Hq,1]
    np.testing.assert_allclose(o, np.broadcast_to(expect, o.shape), rtol=0, atol=1e-13)


def test_window_one_closed_form():
    """W = 1: each query sees only itself, so o_i = v_i * sigmoid(S_ii - sigma)."""
    B, T, Hq, Hkv, D = 1, 25, 4, 2, 8
    q, k, v, sink = _inputs(B, T, Hq, Hkv, D, seed=21)
    scale = 0.7
    o = oracle.prefill(q, k, v, sink, 1, scale)
    qd, kd, vd, sd = (x.double().numpy() for x in (q, k, v, sink))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s_ii = scale * np.einsum("td,td->t", qd[0, :, h], kd[0, :, g])
        w = 1.0 / (1.0 + np.exp(sd[h] - s_ii))
        np.testing.assert_allclose(o[0, :, h], w[:, None] * vd[0, :, g], rtol=0, atol=1e-13)


def test_equal_keys_closed_form():
    """All keys equal: every visible score is the same s, so the output is the
    mean of the visible values times n e^s / (e^sigma + n e^s)."""
    B, T, Hq, Hkv, D, W = 1, 40, 2, 1, 8, 6
    q, _, v, sink = _inputs(B, T, Hq, Hkv, D, seed=4)
    kvec = torch.randn(D, generator=torch.Generator().manual_seed(1))
    k = kvec.expand(B, T, Hkv, D).contiguous()
    scale = 0.25
    o = oracle.prefill(q, k, v, sink, W, scale)
    qd, vd, sd, kd = q.double().numpy(), v.double().numpy(), sink.double().numpy(), kvec.double().numpy()
    for h, i in itertools.product(range(Hq), range(T)):
        lo = max(0, i - W + 1)
        n = i - lo + 1
        s = scale * qd[0, i, h] @ kd
        frac = n * np.exp(s) / (np.exp(sd[h]) + n * np.exp(s))
        np.testing.assert_allclose(o[0, i, h], frac * vd[0, lo:i + 1, 0].mean(0), rtol=0, atol=1e-13)


def test_window_at_least_T_equals_global():
    q, k, v, sink = _inputs(1, 50, 4, 2, 8, seed=8)
    og = oracle.prefill(q, k, v, sink, None, 0.3)
    for window in (50, 51, 1000):
        np.testing.assert_array_equal(oracle.prefill(q, k, v, sink, window, 0.3), og)


def test_rows_subset_equals_full():
    B, T, Hq, Hkv, D = 2, 70, 4, 2, 8
    q, k, v, sink = _inputs(B, T, Hq, Hkv, D, seed=13)
    for window in (None, 9):
        o, lse = oracle.prefill(q, k, v, sink, window, 0.35, want_lse=True)
        rng = np.random.default_rng(0)
        rows = np.stack([rng.integers(0, B, 50), rng.integers(0, T, 50), rng.integers(0, Hq, 50)], 1)
        os_, lses = oracle.prefill_rows(q, k, v, sink, rows, window, 0.35, want_lse=True)
        np.testing.assert_array_equal(os_, o[rows[:, 0], rows[:, 1], rows[:, 2]])
        np.testing.assert_array_equal(lses, lse[rows[:, 0], rows[:, 2], rows[:, 1]])


@pytest.mark.parametrize("window", [None, 4, 128])
def test_verify_equals_brute_force_and_prefill_tail(window):
    """Verify rows: (a) the numpy brute force on the same history; (b) the last
    q_len rows of a prefill over the request's whole sequence, since a draft
    sees exactly the earlier drafts and the history (causal among drafts)."""
    Hq, Hkv, D = 8, 2, 16
    seq_lens = np.array([7, 1, 150, 3], np.int32)
    q_lens = np.array([4, 1, 3, 2], np.int32)
    B, Lmax = len(seq_lens), int(seq_lens.max())
    cu_q = synth.cu_seqlens(q_lens)
    k_hist = synth.normal((B, Lmax, Hkv, D), 1, torch.float32)
    v_hist = synth.normal((B, Lmax, Hkv, D), 2, torch.float32)
    sink = synth.sink_logits(Hq, 3)
    q_full = synth.normal((B, Lmax, Hq, D), 4, torch.float32)
    q = torch.cat([q_full[b, seq_lens[b] - q_lens[b]:seq_lens[b]] for b in range(B)])
    o = oracle.verify(q, cu_q, k_hist, v_hist, seq_lens, sink, window)
    ob = brute.verify(q.numpy(), cu_q, k_hist.numpy(), v_hist.numpy(), seq_lens, sink.numpy(),
                      window, 1.0 / math.sqrt(D))
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    for b in range(B):
        L = int(seq_lens[b])
        op = oracle.prefill(q_full[b:b + 1, :L], k_hist[b:b + 1, :L], v_hist[b:b + 1, :L], sink, window)
        np.testing.assert_array_equal(o[cu_q[b]:cu_q[b + 1]], op[0, L - q_lens[b]:L])
