"""Gradients of sink attention, by the plain definition in fp64 (test
infrastructure only, like the rest of ``oracle``).

Forward (technical-report summary, "MiMo-V2", sections "MiMo-V2-Flash Model
Architecture" and "Hybrid Sliding Window Attention Architecture": SWA with
W = 128, a learnable per-head sink that joins the softmax denominator and
carries no value): for query row i of head h (kv head g = h // (Hq/Hkv)),

    S_ij = scale <q_i, k_j> for visible j,   lse_i = log(e^sigma_h + sum_j e^S_ij)
    P_ij = e^(S_ij - lse_i),   p_sink,i = e^(sigma_h - lse_i),   O_i = sum_j P_ij v_j.

The sink is trained (its learnability is the point of the section above), so
its gradient belongs to the backward pass.  With D_i = <dO_i, O_i>:

    dP_ij = <dO_i, v_j>,   dS_ij = P_ij (dP_ij - D_i)
    dq_i  = scale sum_j dS_ij k_j
    dk_j  = scale sum_{h in group, i} dS_ij q_i,   dv_j = sum_{h in group, i} P_ij dO_i
    dsigma_h = sum_i p_sink,i (0 - D_i)         (the sink column has value 0)

These are the softmax-Jacobian identities written out; the pins compare them
with central finite differences of the forward oracle and with torch's
autograd on a plain torch forward.
"""
from __future__ import annotations

import numpy as np


def _visible(T: int, window: int | None) -> np.ndarray:
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m = j <= i
    if window is not None and window > 0:
        m &= j > i - window
    return m


def prefill_backward(q, k, v, sink, do, window: int | None, scale: float | None = None):
    """q, do [B,T,Hq,D]; k, v [B,T,Hkv,D]; sink [Hq] -> (dq, dk, dv, dsink) in fp64.
    window None or <= 0: global attention."""
    q, k, v, do = (np.asarray(x, np.float64) for x in (q, k, v, do))
    sink = np.asarray(sink, np.float64)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    vis = _visible(T, window)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dsink = np.zeros(Hq)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            S = scale * q[b, :, h] @ k[b, :, g].T
            S = np.where(vis, S, -np.inf)
            sig = sink[h]
            m = np.maximum(sig, S.max(axis=1))
            if np.isposinf(sig):
                continue                               # P = 0, p_sink = 1, O = 0: no gradient
            ms = np.where(np.isfinite(m), m, 0.0)
            e = np.exp(S - ms[:, None])
            es = np.exp(sig - ms) if np.isfinite(sig) else np.zeros(T)
            z = es + e.sum(axis=1)
            P = e / z[:, None]
            psink = es / z
            O = P @ v[b, :, g]
            Di = np.sum(do[b, :, h] * O, axis=1)
            dP = do[b, :, h] @ v[b, :, g].T
            dS = P * (dP - Di[:, None])
            dq[b, :, h] = scale * dS @ k[b, :, g]
            dk[b, :, g] += scale * dS.T @ q[b, :, h]
            dv[b, :, g] += P.T @ do[b, :, h]
            dsink[h] -= np.sum(psink * Di)
    return dq, dk, dv, dsink


def _rows(qb, kb, vb, sig, dob, rows, window, scale):
    """The definition for selected query rows of one (sequence, head): for
    each row i, P_ij over every key j (0 where j is invisible), O_i, D_i and
    dP_ij = <dO_i, v_j>.  qb, dob [T, D]; kb, vb [T, D] of the kv head."""
    T = kb.shape[0]
    rows = np.asarray(rows)
    j = np.arange(T)[None, :]
    vis = j <= rows[:, None]
    if window is not None and window > 0:
        vis &= j > rows[:, None] - window
    S = np.where(vis, scale * qb[rows] @ kb.T, -np.inf)
    if np.isposinf(sig):                          # P = 0, p_sink = 1, O = 0
        P = np.zeros_like(S)
    else:
        m = np.maximum(sig, S.max(axis=1))
        ms = np.where(np.isfinite(m), m, 0.0)
        e = np.exp(S - ms[:, None])
        es = np.exp(sig - ms) if np.isfinite(sig) else np.zeros(len(rows))
        P = e / (es + e.sum(axis=1))[:, None]
    O = P @ vb
    Di = np.sum(dob[rows] * O, axis=1)
    dP = dob[rows] @ vb.T
    return P, Di, dP


def _f64(x):
    """fp64 copy of a (small) slice; torch tensors are moved to the host."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, np.float64)


def query_row_grads(q, k, v, sink, do, window: int | None, b: int, h: int, rows,
                    scale: float | None = None):
    """dq of the query rows `rows` of sequence b, head h, by the definition
    above (fp64, [len(rows), D]): each row needs only its own softmax, so it
    is computed without the rest of the problem.  Only the (b, h) slices are
    read (q, do [B,T,Hq,D], k, v [B,T,Hkv,D], numpy or torch)."""
    D, Hq, Hkv = q.shape[3], q.shape[2], k.shape[2]
    g = h // (Hq // Hkv)
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    qb, kb, vb, dob = _f64(q[b, :, h]), _f64(k[b, :, g]), _f64(v[b, :, g]), _f64(do[b, :, h])
    P, Di, dP = _rows(qb, kb, vb, float(sink[h]), dob, rows, window, scale)
    dS = P * (dP - Di[:, None])
    return scale * dS @ kb


def key_row_grads(q, k, v, sink, do, window: int | None, b: int, g: int, keys,
                  scale: float | None = None):
    """dk and dv of the keys `keys` of sequence b, kv head g, by the
    definition above (fp64, two [len(keys), D] arrays): the sums over the
    query rows that see them (rows min(keys) .. the last row that sees
    max(keys)) of every query head of the group."""
    T, Hq, D = q.shape[1], q.shape[2], q.shape[3]
    G = Hq // k.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    keys = np.asarray(keys)
    last = T - 1
    if window is not None and window > 0:
        last = min(last, int(keys.max()) + window - 1)
    rows = np.arange(int(keys.min()), last + 1)
    kb, vb = _f64(k[b, :, g]), _f64(v[b, :, g])
    dk = np.zeros((len(keys), D))
    dv = np.zeros((len(keys), D))
    for h in range(g * G, (g + 1) * G):
        qb, dob = _f64(q[b, :, h]), _f64(do[b, :, h])
        P, Di, dP = _rows(qb, kb, vb, float(sink[h]), dob, rows, window, scale)
        dS = P * (dP - Di[:, None])
        dk += scale * dS[:, keys].T @ qb[rows]
        dv += P[:, keys].T @ dob[rows]
    return dk, dv
