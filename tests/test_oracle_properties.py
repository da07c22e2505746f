"""Property-based pins of the C oracle against the numpy brute force (a second
formulation: full score matrix, -inf outside the mask, an appended sink column,
scipy softmax) over many small random configurations: batch, length (ragged,
including 1), GQA group size, head dim, window (including 1 and >= T), scale,
and sink logits drawn from finite values and +-inf; prefill and verify (random
history lengths and 1..4 draft rows).  The oracle's gradients are checked the
same way against torch's fp64 autograd of a plain torch forward.  Examples are
derandomized, so every run checks the same cases.  CPU only."""
import math

import numpy as np
import pytest
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle
from oracle import brute

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True,
                    suppress_health_check=[HealthCheck.too_slow])

sink_values = st.one_of(st.floats(-6.0, 6.0), st.sampled_from([math.inf, -math.inf]))


@st.composite
def prefill_case(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 24))
    Hkv = draw(st.sampled_from([1, 2]))
    G = draw(st.sampled_from([1, 2, 4]))
    D = draw(st.sampled_from([4, 8]))
    window = draw(st.one_of(st.none(), st.integers(1, 30)))
    scale = draw(st.sampled_from([None, 0.05, 1.0]))
    sinks = draw(st.lists(sink_values, min_size=Hkv * G, max_size=Hkv * G))
    seed = draw(st.integers(0, 2**31 - 1))
    return B, T, Hkv * G, Hkv, D, window, scale, sinks, seed


@SETTINGS
@given(prefill_case())
def test_prefill_oracle_equals_brute_force(case):
    B, T, Hq, Hkv, D, window, scale, sinks, seed = case
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    sink = np.asarray(sinks, np.float32)
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    o, lse, ps = oracle.prefill(q, k, v, sink, window, sc, want_lse=True, want_psink=True)
    ob, psb, lseb = brute.prefill(q, k, v, sink, window, sc)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-11)
    np.testing.assert_allclose(ps, psb, rtol=0, atol=1e-11)
    fin = np.isfinite(lseb)
    assert np.array_equal(fin, np.isfinite(lse)) and np.array_equal(lse[~fin], lseb[~fin])
    np.testing.assert_allclose(lse[fin], lseb[fin], rtol=1e-12, atol=1e-11)


@st.composite
def verify_case(draw):
    B = draw(st.integers(1, 3))
    Hkv = draw(st.sampled_from([1, 2]))
    G = draw(st.sampled_from([1, 4]))
    D = draw(st.sampled_from([4, 8]))
    q_lens = draw(st.lists(st.integers(1, 4), min_size=B, max_size=B))
    extra = draw(st.lists(st.integers(0, 40), min_size=B, max_size=B))
    window = draw(st.one_of(st.none(), st.integers(1, 20)))
    sinks = draw(st.lists(sink_values, min_size=Hkv * G, max_size=Hkv * G))
    seed = draw(st.integers(0, 2**31 - 1))
    return Hkv * G, Hkv, D, q_lens, extra, window, sinks, seed


@SETTINGS
@given(verify_case())
def test_verify_oracle_equals_brute_force(case):
    Hq, Hkv, D, q_lens, extra, window, sinks, seed = case
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray([ql + e for ql, e in zip(q_lens, extra)], np.int32)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    B, Lmax = len(q_lens), int(seq_lens.max())
    q = rng.standard_normal((int(cu_q[-1]), Hq, D)).astype(np.float32)
    k_hist = rng.standard_normal((B, Lmax, Hkv, D)).astype(np.float32)
    v_hist = rng.standard_normal((B, Lmax, Hkv, D)).astype(np.float32)
    sink = np.asarray(sinks, np.float32)
    sc = 1.0 / math.sqrt(D)
    o = oracle.verify(q, cu_q, k_hist, v_hist, seq_lens, sink, window, sc)
    ob = brute.verify(q, cu_q, k_hist, v_hist, seq_lens, sink, window, sc)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-11)


@st.composite
def backward_case(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 12))
    Hkv = draw(st.sampled_from([1, 2]))
    G = draw(st.sampled_from([1, 2, 4]))
    D = draw(st.sampled_from([4, 8]))
    window = draw(st.one_of(st.none(), st.integers(1, 14)))
    sinks = draw(st.lists(st.one_of(st.floats(-4.0, 4.0), st.just(-math.inf)),
                          min_size=Hkv * G, max_size=Hkv * G))
    seed = draw(st.integers(0, 2**31 - 1))
    return B, T, Hkv * G, Hkv, D, window, sinks, seed


@settings(max_examples=40, deadline=None, derandomize=True,
          suppress_health_check=[HealthCheck.too_slow])
@given(backward_case())
def test_backward_oracle_equals_torch_autograd(case):
    """The oracle's gradients (dq, dk, dv, dsink) against torch's fp64 autograd
    of a plain torch forward (masked scores, a sink column, library softmax)."""
    import torch
    from oracle import backward
    B, T, Hq, Hkv, D, window, sinks, seed = case
    rng = np.random.default_rng(seed)
    q, do = (rng.standard_normal((B, T, Hq, D)) for _ in range(2))
    k, v = (rng.standard_normal((B, T, Hkv, D)) for _ in range(2))
    sink = np.asarray(sinks, np.float64)
    ours = backward.prefill_backward(q, k, v, sink, do, window)
    tq, tk, tv, ts = (torch.tensor(x, requires_grad=True) for x in (q, k, v, sink))
    G = Hq // Hkv
    s = torch.einsum("bihd,bjhd->bhij", tq, tk.repeat_interleave(G, dim=2)) / math.sqrt(D)
    i, j = torch.arange(T)[:, None], torch.arange(T)[None, :]
    vis = (j <= i) & ((j > i - window) if window else torch.ones(T, T, dtype=torch.bool))
    s = s.masked_fill(~vis, -math.inf)
    col = ts.view(1, Hq, 1, 1).expand(B, Hq, T, 1)
    p = torch.softmax(torch.cat([s, col], dim=-1), dim=-1)[..., :T]
    o = torch.einsum("bhij,bjhd->bihd", p, tv.repeat_interleave(G, dim=2))
    (o * torch.tensor(do)).sum().backward()
    ref = (tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(), ts.grad.numpy())
    for name, a, b in zip(("dq", "dk", "dv", "dsink"), ours, ref):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11, err_msg=name)
