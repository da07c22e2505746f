"""Backward parity: attn_sink_prefill_backward (through the C ABI) against
oracle.backward.prefill_backward in fp64 on the same bf16 inputs, for the
sliding window (W = 128 and a smaller one), global attention, GQA, ragged
tile tails and infinite sinks.

Tolerance.  The kernel rounds P and dS to bf16 before the products that use
them, as the forward rounds P; each gradient element is a sum of many such
terms, so the error of dq, dk, dv is measured relative to the size of the
gradient: relative L2 <= 1e-2 and max-abs <= 2e-2 * max|reference|.  dsink is
an fp32 sum over all rows of a head: relative error <= 1e-2 of its scale."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import errors
from oracle import backward

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS_FRAC = 2e-2


def _close(out, ref, what):
    out = out.detach().float().cpu().double().numpy()
    assert np.isfinite(out).all(), f"{what}: non-finite"
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    max_abs, rel = errors(out, ref)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e}"
    assert max_abs <= MAX_ABS_FRAC * scale, f"{what}: max-abs {max_abs:.3e} vs scale {scale:.3e}"
    return rel


def _run(B, T, Hq, Hkv, window, seed, sink_override=None):
    q, k, v, sink = synth.prefill_inputs(B, T, Hq, Hkv, 128, seed)
    if sink_override is not None:
        for h, s in sink_override.items():
            sink[h] = s
    dout = synth.normal((B, T, Hq, 128), seed + 1)
    qd, kd, vd, sd, dod = q.cuda(), k.cuda(), v.cuda(), sink.cuda(), dout.cuda()
    lse = torch.empty(B, Hq, T, device="cuda")
    if window:
        o = A.attn_swa_sink_prefill(qd, kd, vd, sd, window=window, lse=lse)
    else:
        o = A.attn_ga_sink_prefill(qd, kd, vd, sd, lse=lse)
    dq, dk, dv, ds = A.attn_sink_prefill_backward(qd, kd, vd, o, lse, dod, sd, window=window)
    assert A.attn_check_device_error() == 0
    ref = backward.prefill_backward(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                    sink.numpy(), dout.float().numpy(), window or None)
    return (dq, dk, dv, ds), ref


@pytest.mark.parametrize("B,T,Hq,Hkv,window", [
    (1, 200, 16, 2, 128), (2, 77, 8, 1, 64), (1, 300, 8, 8, 0), (1, 1, 8, 2, 128),
    (1, 129, 64, 8, 128), (1, 513, 8, 1, 128),
    # more query-tile items than CTAs: each persistent CTA reuses its TMEM Q/dO
    # copy and its dQ accumulator across items
    (1, 1100, 32, 4, 128), (1, 700, 32, 4, 0),
])
def test_backward_matches_oracle(B, T, Hq, Hkv, window):
    got, ref = _run(B, T, Hq, Hkv, window, seed=T + Hq)
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        _close(g, r, f"{name} T={T} W={window}")
    ds = got[3].cpu().double().numpy()
    assert np.max(np.abs(ds - ref[3])) <= 1e-2 * max(np.max(np.abs(ref[3])), 1e-3)


def test_backward_infinite_sinks():
    got, ref = _run(1, 150, 8, 2, 128, seed=9, sink_override={0: math.inf, 3: -math.inf})
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        _close(g, r, f"{name} inf sinks")
    ds = got[3].cpu().double().numpy()
    assert ds[0] == 0.0 and ds[3] == 0.0
    assert np.max(np.abs(ds - ref[3])) <= 1e-2 * max(np.max(np.abs(ref[3])), 1e-3)
    assert not got[0][:, :, 0].float().abs().max().item()  # head 0 (sigma = +inf): dq = 0


def test_full_size_backward_prefix_rows():
    """T = 32768, Hq = 64, Hkv = 8, W = 128: the gradients of the first L rows'
    queries and of keys j < L - W depend on rows < L only, so they must equal
    the oracle on the length-L prefix of the same inputs."""
    T, L, W = 32768, 384, 128
    q, k, v, sink = synth.prefill_inputs(1, T, 64, 8, 128, 1008, device="cuda")
    dout = synth.normal((1, T, 64, 128), 1009, device="cuda")
    lse = torch.empty(1, 64, T, device="cuda")
    o = A.attn_swa_sink_prefill(q, k, v, sink, window=W, lse=lse)
    dq, dk, dv, _ = A.attn_sink_prefill_backward(q, k, v, o, lse, dout, sink, window=W)
    assert A.attn_check_device_error() == 0
    ref = backward.prefill_backward(q[:, :L].float().cpu().numpy(), k[:, :L].float().cpu().numpy(),
                                    v[:, :L].float().cpu().numpy(), sink.cpu().numpy(),
                                    dout[:, :L].float().cpu().numpy(), W)
    _close(dq[:, :L], ref[0], "full-size dq prefix")
    _close(dk[:, :L - W], ref[1][:, :L - W], "full-size dk prefix")
    _close(dv[:, :L - W], ref[2][:, :L - W], "full-size dv prefix")


def _full_size_run(window, seed):
    T = 32768
    q, k, v, sink = synth.prefill_inputs(1, T, 64, 8, 128, seed, device="cuda")
    dout = synth.normal((1, T, 64, 128), seed + 1, device="cuda")
    lse = torch.empty(1, 64, T, device="cuda")
    if window:
        o = A.attn_swa_sink_prefill(q, k, v, sink, window=window, lse=lse)
    else:
        o = A.attn_ga_sink_prefill(q, k, v, sink, lse=lse)
    dq, dk, dv, _ = A.attn_sink_prefill_backward(q, k, v, o, lse, dout, sink, window=window)
    assert A.attn_check_device_error() == 0
    return (q, k, v, sink.cpu().numpy(), dout), (dq, dk, dv)


@pytest.mark.parametrize("window", [0, 128])
def test_full_size_backward_sampled_rows_and_keys(window):
    """T = 32768, Hq = 64, Hkv = 8: dq of sampled query rows (each needs only
    its own softmax) and dk, dv of sampled keys (sums over the rows that see
    them) against the oracle's row and key gradients.  Under global attention
    the keys are the last ones, whose rows the oracle can still afford."""
    T = 32768
    (q, k, v, sink, dout), (dq, dk, dv) = _full_size_run(window, 1010 + window)
    rows = np.array([0, 1, 4097, T // 2 + 3, T - 1])
    got, ref = [], []
    for h in (0, 37, 63):
        got.append(dq[0, rows, h].float().cpu().numpy())
        ref.append(backward.query_row_grads(q, k, v, sink, dout, window or None, 0, h, rows))
    _close(torch.from_numpy(np.concatenate(got)), np.concatenate(ref), f"dq rows W={window}")
    # clusters of keys, so the rows that see them stay few
    clusters = ([np.array([T - 200, T - 77, T - 1])] if not window
                else [np.array([5, 9]), np.array([16000, 16001, 16100]), np.array([T - 3, T - 1])])
    gk, gv, rk, rv = [], [], [], []
    for g in (0, 7):
        for keys in clusters:
            a, c = backward.key_row_grads(q, k, v, sink, dout, window or None, 0, g, keys)
            rk.append(a)
            rv.append(c)
            gk.append(dk[0, keys, g].float().cpu().numpy())
            gv.append(dv[0, keys, g].float().cpu().numpy())
    _close(torch.from_numpy(np.concatenate(gk)), np.concatenate(rk), f"dk keys W={window}")
    _close(torch.from_numpy(np.concatenate(gv)), np.concatenate(rv), f"dv keys W={window}")
