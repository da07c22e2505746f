"""Pins of the oracle's gradients (oracle.backward.prefill_backward) against
things other than themselves: central finite differences of the C forward
oracle in fp64, and torch's autograd (fp64) of a plain torch forward (masked
scores plus a sink column, a library softmax, the sink column dropped).
Planted mistakes must fail.  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import backward

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(B, T, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, D))
    k = rng.standard_normal((B, T, Hkv, D))
    v = rng.standard_normal((B, T, Hkv, D))
    sink = rng.standard_normal(Hq)
    do = rng.standard_normal((B, T, Hq, D))
    return q, k, v, sink, do


def _fd(fn, x, eps=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + eps
        fp = fn()
        x[idx] = old - eps
        fm = fn()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * eps)
    return g


def _torch_grads(q, k, v, sink, do, window):
    tq, tk, tv, ts = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v, sink))
    B, T, Hq, D = q.shape
    G = Hq // k.shape[2]
    kk = tk.repeat_interleave(G, dim=2)
    vv = tv.repeat_interleave(G, dim=2)
    S = torch.einsum("bihd,bjhd->bhij", tq, kk) / math.sqrt(D)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    vis = j <= i
    if window:
        vis &= j > i - window
    S = S.masked_fill(~vis, float("-inf"))
    col = ts.view(1, Hq, 1, 1).expand(B, Hq, T, 1)
    P = torch.softmax(torch.cat([S, col], dim=-1), dim=-1)[..., :T]
    O = torch.einsum("bhij,bjhd->bihd", P, vv)
    (O * torch.tensor(do)).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(), ts.grad.numpy()


@pytest.mark.parametrize("window", [None, 3])
def test_matches_finite_differences_of_the_forward_oracle(window):
    q, k, v, sink, do = _inputs(1, 7, 4, 2, 4, 1)

    def loss():
        o = oracle.prefill(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32),
                           sink.astype(np.float32), window)
        return float(np.sum(o * do))
    # the C oracle takes fp32 inputs: step on values that fp32 holds exactly
    for x in (q, k, v, sink):
        x[...] = x.astype(np.float32)
    dq, dk, dv, ds = backward.prefill_backward(q, k, v, sink, do, window)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv), ("sink", sink, ds)):
        num = _fd(loss, x, eps=1e-3)
        np.testing.assert_allclose(g, num, rtol=2e-3, atol=2e-4, err_msg=name)


@pytest.mark.parametrize("B,T,Hq,Hkv,D,window", [(2, 9, 4, 2, 8, None), (1, 13, 8, 2, 4, 4),
                                                 (1, 6, 2, 1, 16, 1)])
def test_matches_torch_autograd(B, T, Hq, Hkv, D, window):
    q, k, v, sink, do = _inputs(B, T, Hq, Hkv, D, 2 + T)
    ours = backward.prefill_backward(q, k, v, sink, do, window)
    ref = _torch_grads(q, k, v, sink, do, window)
    for name, a, b in zip(("dq", "dk", "dv", "dsink"), ours, ref):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12, err_msg=name)


def test_infinite_sinks():
    q, k, v, sink, do = _inputs(1, 5, 2, 1, 4, 3)
    sink[:] = [math.inf, -math.inf]
    dq, dk, dv, ds = backward.prefill_backward(q, k, v, sink, do, None)
    assert not dq[:, :, 0].any() and ds[0] == 0.0 and ds[1] == 0.0
    ref = _torch_grads(q, k, v, np.array([-30.0, -math.inf]), do, None)  # head 1: plain softmax
    np.testing.assert_allclose(dq[:, :, 1], ref[0][:, :, 1], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mutant", ["sink_sign", "dk_unscaled", "dv_uses_dP", "D_from_q"])
def test_pins_reject_planted_mistakes(mutant, monkeypatch):
    orig = backward.prefill_backward

    def bad(q, k, v, sink, do, window, scale=None):
        dq, dk, dv, ds = orig(q, k, v, sink, do, window, scale)
        if mutant == "sink_sign":
            ds = -ds
        elif mutant == "dk_unscaled":
            dk = dk * math.sqrt(q.shape[-1])
        elif mutant == "dv_uses_dP":
            dv = dv + 0.01
        elif mutant == "D_from_q":
            dq = dq * 1.01
        return dq, dk, dv, ds
    monkeypatch.setattr(backward, "prefill_backward", bad)
    with pytest.raises(AssertionError):
        test_matches_torch_autograd(1, 9, 4, 2, 8, 3)


@pytest.mark.parametrize("B,T,Hq,Hkv,window,sinks", [
    (1, 40, 4, 1, 8, None), (2, 33, 4, 2, None, None), (1, 50, 8, 2, 1, None),
    (1, 37, 2, 1, 100, {0: math.inf, 1: -math.inf}),
])
def test_sampled_row_and_key_gradients_equal_the_full_backward(B, T, Hq, Hkv, window, sinks):
    """query_row_grads / key_row_grads (used for full-size checks, where the
    full backward is out of reach) give exactly the rows of prefill_backward."""
    q, k, v, sink, do = _inputs(B, T, Hq, Hkv, 16, seed=T + Hq)
    for hh, s in (sinks or {}).items():
        sink[hh] = s
    dq, dk, dv, _ = backward.prefill_backward(q, k, v, sink, do, window)
    rows = np.array([0, 1, T // 2, T - 1])
    keys = np.array([0, 3, T - 5, T - 1])
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(backward.query_row_grads(q, k, v, sink, do, window, b, h, rows),
                                       dq[b, rows, h], rtol=1e-10, atol=1e-12)
        for g in range(Hkv):
            gk, gv = backward.key_row_grads(q, k, v, sink, do, window, b, g, keys)
            np.testing.assert_allclose(gk, dk[b, keys, g], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(gv, dv[b, keys, g], rtol=1e-10, atol=1e-12)
