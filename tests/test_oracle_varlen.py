"""Pins of the oracle's packed-batch prefill (oracle.prefill_varlen) against
things other than itself: the numpy brute force applied to each sequence on
its own (a second formulation), the batched oracle on equal lengths (a fixed
layout: o [total,Hq,D] = o[B,T] flattened, lse [Hq,total] = lse[B,Hq,T]
transposed), independence of the sequences (changing one sequence's tokens
leaves every other output unchanged), and linearity in value_scale (o scales,
lse does not).  Each pin also runs against plausible mistakes planted in a
copy of the function here on the CPU, and must reject every one of them.
CPU only.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import brute

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _packed(lens, Hq, Hkv, D, seed):
    total = int(sum(lens))
    q, k, v, sink = synth.prefill_inputs(1, max(total, 1), Hq, Hkv, D, seed, dtype=torch.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q[0, :total], k[0, :total], v[0, :total], sink, cu


# ------------------------------------------------------------------ pins
def pin_brute_force(fn):
    lens, Hq, Hkv, D = [5, 0, 17, 1, 9], 4, 2, 8
    q, k, v, sink, cu = _packed(lens, Hq, Hkv, D, 11)
    sink = torch.tensor([0.5, -math.inf, 2.0, -1.0])
    for window in (None, 4):
        o, lse = fn(q, k, v, cu, sink, window, want_lse=True)
        for b in range(len(lens)):
            s, e = cu[b], cu[b + 1]
            if e == s:
                continue
            ob, _, lb = brute.prefill(q[None, s:e].numpy().astype(np.float64),
                                      k[None, s:e].numpy().astype(np.float64),
                                      v[None, s:e].numpy().astype(np.float64),
                                      sink.numpy().astype(np.float64), window, 1 / math.sqrt(D))
            if not (np.allclose(o[s:e], ob[0], atol=1e-10) and np.allclose(lse[:, s:e], lb[0], atol=1e-10)):
                return False
    return True


def pin_equal_lengths_equal_the_batched_layout(fn):
    B, T, Hq, Hkv, D = 3, 13, 4, 2, 8
    q, k, v, sink = synth.prefill_inputs(B, T, Hq, Hkv, D, 12, dtype=torch.float32)
    cu = np.arange(B + 1, dtype=np.int32) * T
    ob, lb = oracle.prefill(q, k, v, sink, 5, want_lse=True)
    o, lse = fn(q.reshape(B * T, Hq, D), k.reshape(B * T, Hkv, D), v.reshape(B * T, Hkv, D), cu,
                sink, 5, want_lse=True)
    return (np.array_equal(o, ob.reshape(B * T, Hq, D)) and
            np.array_equal(lse, lb.transpose(1, 0, 2).reshape(Hq, B * T)))


def pin_sequences_are_independent(fn):
    lens, Hq, Hkv, D = [7, 12, 3], 4, 2, 8
    q, k, v, sink, cu = _packed(lens, Hq, Hkv, D, 13)
    o = fn(q, k, v, cu, sink, None)
    k2, v2 = k.clone(), v.clone()
    k2[cu[1]:cu[2]] += 1.0   # change sequence 1 only
    v2[cu[1]:cu[2]] -= 2.0
    o2 = fn(q, k2, v2, cu, sink, None)
    others = np.r_[cu[0]:cu[1], cu[2]:cu[3]]
    return np.array_equal(o[others], o2[others]) and not np.allclose(o[cu[1]:cu[2]], o2[cu[1]:cu[2]])


def pin_value_scale_is_linear(fn):
    lens, Hq, Hkv, D = [6, 10], 4, 1, 8
    q, k, v, sink, cu = _packed(lens, Hq, Hkv, D, 14)
    o1, l1 = fn(q, k, v, cu, sink, 3, want_lse=True)
    o2, l2 = fn(q, k, v, cu, sink, 3, value_scale=0.707, want_lse=True)
    return np.allclose(o2, 0.707 * o1, rtol=1e-14, atol=0) and np.array_equal(l1, l2)


PINS = [pin_brute_force, pin_equal_lengths_equal_the_batched_layout,
        pin_sequences_are_independent, pin_value_scale_is_linear]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_varlen_pin(pin):
    assert pin(oracle.prefill_varlen)


# --------------------------------------------------------------- mutants
def _mutant(kind):
    def fn(q, k, v, cu_seqlens, sink, window, scale=None, value_scale=1.0, want_lse=False):
        q, k, v, sink = (np.asarray(t, np.float32) for t in (q, k, v, sink))
        cu = np.asarray(cu_seqlens, np.int32)
        total, Hq, D = q.shape
        o = np.zeros((total, Hq, D))
        lse = np.zeros((Hq, total))
        for b in range(len(cu) - 1):
            s, e = int(cu[b]), int(cu[b + 1])
            if kind == "one_token_of_history":   # the previous sequence's last key leaks in
                s_k = max(s - 1, 0)
            else:
                s_k = s
            if e == s:
                continue
            qs = q[None, s:e]
            ks, vs = k[None, s_k:e], v[None, s_k:e]
            if kind == "one_token_of_history" and s_k < s:
                qs = np.concatenate([q[None, s_k:s_k + 1], qs], axis=1)
            ob, lb = oracle.prefill(qs, ks, vs, sink, window, scale, want_lse=True)
            off = ob.shape[1] - (e - s)
            o[s:e] = ob[0, off:]
            lse[:, s:e] = lb[0, :, off:]
            if kind == "scale_also_lse":
                lse[:, s:e] += math.log(value_scale)
            if kind != "scale_dropped":
                o[s:e] *= value_scale
        if kind == "lse_sequence_major":   # [B,Hq,len] blocks instead of [Hq,total]
            lse = lse.T.reshape(Hq, total) if total % Hq == 0 else lse[::-1]
        return (o, lse) if want_lse else o
    return fn


@pytest.mark.parametrize("kind", ["one_token_of_history", "scale_also_lse", "scale_dropped",
                                  "lse_sequence_major"])
def test_pins_reject_planted_mistakes(kind):
    fn = _mutant(kind)
    assert not all(pin(fn) for pin in PINS), kind
