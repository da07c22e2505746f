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
