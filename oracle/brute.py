"""Brute-force numpy formulation of sink attention (tiny inputs only).

TEST INFRASTRUCTURE ONLY.  A second, independent way of writing the same
definition as the C oracle, used to pin it: build the whole score matrix,
put -inf outside the mask, append the sink logit as one more column, take a
library softmax over the row, drop the sink column and multiply by V.  The
sink column has no value vector, so it only enlarges the denominator
(MiMo-V2-Flash technical-report summary, section "Hybrid Sliding Window
Attention Architecture": learnable gpt-oss-style sink bias).
"""
from __future__ import annotations

import numpy as np
from scipy.special import softmax


def mask_matrix(Tq: int, Tk: int, q_pos: np.ndarray, window: int | None) -> np.ndarray:
    """allowed[r, j] for query positions q_pos[r] and key positions 0..Tk-1."""
    j = np.arange(Tk)[None, :]
    i = np.asarray(q_pos)[:, None]
    allowed = j <= i
    if window is not None and window > 0:
        allowed &= j > i - window
    return allowed


def _rows(qh, kh, vh, q_pos, sigma, window, scale):
    """qh [n,D], kh/vh [Tk,D] (fp64).  Returns o [n,D], p_sink [n], lse [n]."""
    n, Tk = qh.shape[0], kh.shape[0]
    S = scale * (qh @ kh.T)
    S = np.where(mask_matrix(n, Tk, q_pos, window), S, -np.inf)
    if np.isposinf(sigma):
        return np.zeros((n, vh.shape[1])), np.ones(n), np.full(n, np.inf)
    ext = np.concatenate([S, np.full((n, 1), sigma)], axis=1)
    P = softmax(ext, axis=1)
    m = np.max(ext, axis=1)
    lse = m + np.log(np.sum(np.exp(ext - m[:, None]), axis=1))
    return P[:, :Tk] @ vh, P[:, Tk], lse


def prefill(q, k, v, sink, window, scale):
    """q [B,T,Hq,D], k/v [B,T,Hkv,D] -> o [B,T,Hq,D], p_sink [B,Hq,T], lse [B,Hq,T]."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    sink = np.asarray(sink, np.float64)
    B, T, Hq, D = q.shape
    G = Hq // k.shape[2]
    o = np.zeros_like(q)
    ps = np.zeros((B, Hq, T))
    lse = np.zeros((B, Hq, T))
    for b in range(B):
        for h in range(Hq):
            g = h // G
            o[b, :, h], ps[b, h], lse[b, h] = _rows(q[b, :, h], k[b, :, g], v[b, :, g],
                                                    np.arange(T), sink[h], window, scale)
    return o, ps, lse


def verify(q, cu_q, k_hist, v_hist, seq_lens, sink, window, scale):
    """Verify rows against a linear history (see the C oracle for layouts)."""
    q, k_hist, v_hist = (np.asarray(x, np.float64) for x in (q, k_hist, v_hist))
    sink = np.asarray(sink, np.float64)
    nq, Hq, D = q.shape
    B = k_hist.shape[0]
    G = Hq // k_hist.shape[2]
    o = np.zeros_like(q)
    for b in range(B):
        r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
        L = int(seq_lens[b])
        pos = np.arange(L - (r1 - r0), L)
        for h in range(Hq):
            g = h // G
            o[r0:r1, h], _, _ = _rows(q[r0:r1, h], k_hist[b, :L, g], v_hist[b, :L, g],
                                      pos, sink[h], window, scale)
    return o
