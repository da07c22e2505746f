"""Sink-attention oracle (fp64, CPU).

TEST INFRASTRUCTURE ONLY: tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never
does.  It shares no code with the CUDA library in
``global_attention_sinks_swa_b300`` and imports nothing from it.

Contents
--------
- ``prefill`` / ``prefill_rows`` / ``verify``: ctypes wrappers over the plain C
  implementation in ``attn_sink_oracle.c`` (fp64 loops, OpenMP over rows);
  ``prefill_varlen`` applies ``prefill`` to each sequence of a packed batch.
- ``brute``: a second formulation in numpy (full score matrix, an appended sink
  column, a library softmax) used to pin the C code on tiny inputs.
- ``index``: the integer definitions the kernels' index arithmetic must
  reproduce bit for bit (visibility, ring slot, page location).
- ``backward``: gradients dq, dk, dv and the sink's dsigma by the softmax
  Jacobian written out in fp64.
- ``fp8``: the E4M3 codes of an 8-bit KV cache (decode, encode with
  round-to-nearest-even and saturation, per-kv-head scales); ``verify_fp8``
  is ``verify`` over the dequantized history.

Method sources: MiMo-V2-Flash technical-report summary (fanfer.top,
"MiMo-V2"), sections "MiMo-V2-Flash Model Architecture" (W = 128, 5:1 hybrid)
and "Hybrid Sliding Window Attention Architecture" (learnable gpt-oss-style
sink bias); release announcement (aihot.news, "小米开源 MiMo-V2-Flash"),
section "将效率推向极限" (fixed-size SWA KV cache) and figure
"Multi-Token Prediction" (verify 1 + 3 drafts, accept a prefix).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import backward, brute, fp8, index  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_sink_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (the checker is built, never shipped)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
            f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
            i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
            vp = ctypes.c_void_p
            ci, cd, cl = ctypes.c_int, ctypes.c_double, ctypes.c_long
            lib.oracle_prefill.argtypes = [f32p, f32p, f32p, f32p, f64p, vp, vp,
                                           ci, ci, ci, ci, ci, ci, cd]
            lib.oracle_prefill_rows.argtypes = [f32p, f32p, f32p, f32p, i32p, cl, f64p, vp, vp,
                                                ci, ci, ci, ci, ci, ci, cd]
            lib.oracle_verify.argtypes = [f32p, i32p, f32p, f32p, ci, i32p, f32p, f64p, vp, vp,
                                          ci, ci, ci, ci, ci, cd]
            for fn in (lib.oracle_prefill, lib.oracle_prefill_rows, lib.oracle_verify):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    """Widen to a contiguous fp32 numpy array (bf16 -> fp32 is exact)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _i32(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_scale(D: int) -> float:
    return 1.0 / float(np.sqrt(D))


def prefill(q, k, v, sink, window: int | None, scale: float | None = None,
            want_lse: bool = False, want_psink: bool = False):
    """Prefill by the plain definition.  q [B,T,Hq,D], k/v [B,T,Hkv,D],
    sink [Hq]; ``window=None`` (or <= 0) selects global attention.
    Returns o (fp64 [B,T,Hq,D]) and, on request, lse / psink ([B,Hq,T])."""
    q, k, v, sink = _f32(q), _f32(k), _f32(v), _f32(sink)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, T, Hkv, D) or v.shape != k.shape or sink.shape != (Hq,):
        raise ValueError("oracle.prefill: inconsistent shapes")
    scale = default_scale(D) if scale is None else float(scale)
    o = np.zeros((B, T, Hq, D), np.float64)
    lse = np.zeros((B, Hq, T), np.float64) if want_lse else None
    ps = np.zeros((B, Hq, T), np.float64) if want_psink else None
    rc = _load().oracle_prefill(q, k, v, sink, o, _ptr(lse), _ptr(ps),
                                B, T, Hq, Hkv, D, int(window or 0), scale)
    if rc != 0:
        raise ValueError("oracle_prefill rejected its arguments")
    out = [o] + ([lse] if want_lse else []) + ([ps] if want_psink else [])
    return out[0] if len(out) == 1 else tuple(out)


def prefill_rows(q, k, v, sink, rows, window: int | None, scale: float | None = None,
                 want_lse: bool = False):
    """Selected rows of the prefill, rows = int array [n, 3] of (b, i, h).
    Returns o [n, D] (and lse [n])."""
    q, k, v, sink = _f32(q), _f32(k), _f32(v), _f32(sink)
    rows = _i32(rows).reshape(-1, 3)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    scale = default_scale(D) if scale is None else float(scale)
    n = rows.shape[0]
    o = np.zeros((n, D), np.float64)
    lse = np.zeros((n,), np.float64) if want_lse else None
    rc = _load().oracle_prefill_rows(q, k, v, sink, rows, n, o, _ptr(lse), None,
                                     B, T, Hq, Hkv, D, int(window or 0), scale)
    if rc != 0:
        raise ValueError("oracle_prefill_rows rejected its arguments")
    return (o, lse) if want_lse else o


def prefill_varlen(q, k, v, cu_seqlens, sink, window: int | None, scale: float | None = None,
                   value_scale: float = 1.0, want_lse: bool = False):
    """Prefill of a packed batch: q [total,Hq,D], k/v [total,Hkv,D], sequence b
    = tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 with positions 0..len-1, each
    sequence attending only to itself (the plain definition per sequence).
    The output is multiplied by value_scale: the reading of the model
    configuration's attention_value_scale (dpshk.com article on
    MiMo-V2-Flash-Base, section "轻量级多token预测技术") as a factor on the
    attention output; the LSE is unscaled.
    Returns o (fp64 [total,Hq,D]) and, on request, lse (fp64 [Hq,total])."""
    q, k, v, sink = _f32(q), _f32(k), _f32(v), _f32(sink)
    cu = _i32(cu_seqlens)
    total, Hq, D = q.shape
    if (cu.ndim != 1 or cu.shape[0] < 1 or cu[0] != 0 or cu[-1] != total
            or np.any(np.diff(cu) < 0) or k.shape[0] != total or v.shape != k.shape):
        raise ValueError("oracle.prefill_varlen: inconsistent shapes or offsets")
    o = np.zeros((total, Hq, D), np.float64)
    lse = np.zeros((Hq, total), np.float64)
    for b in range(cu.shape[0] - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        if e == s:
            continue
        ob, lb = prefill(q[None, s:e], k[None, s:e], v[None, s:e], sink, window, scale,
                         want_lse=True)
        o[s:e] = float(value_scale) * ob[0]
        lse[:, s:e] = lb[0]
    return (o, lse) if want_lse else o


def verify(q, cu_q, k_hist, v_hist, seq_lens, sink, window: int | None,
           scale: float | None = None, want_lse: bool = False, want_psink: bool = False):
    """MTP verify by the plain definition on a linear history.
    q [sum_q,Hq,D], cu_q [B+1], k_hist/v_hist [B,Lmax,Hkv,D], seq_lens [B]."""
    q, k_hist, v_hist, sink = _f32(q), _f32(k_hist), _f32(v_hist), _f32(sink)
    cu_q, seq_lens = _i32(cu_q), _i32(seq_lens)
    nq, Hq, D = q.shape
    B, Lmax, Hkv, _ = k_hist.shape
    if cu_q.shape != (B + 1,) or seq_lens.shape != (B,) or cu_q[-1] != nq:
        raise ValueError("oracle.verify: inconsistent shapes")
    scale = default_scale(D) if scale is None else float(scale)
    o = np.zeros((nq, Hq, D), np.float64)
    lse = np.zeros((nq, Hq), np.float64) if want_lse else None
    ps = np.zeros((nq, Hq), np.float64) if want_psink else None
    rc = _load().oracle_verify(q, cu_q, k_hist, v_hist, Lmax, seq_lens, sink, o,
                               _ptr(lse), _ptr(ps), B, Hq, Hkv, D, int(window or 0), scale)
    if rc != 0:
        raise ValueError("oracle_verify rejected its arguments")
    out = [o] + ([lse] if want_lse else []) + ([ps] if want_psink else [])
    return out[0] if len(out) == 1 else tuple(out)


def verify_fp8(q, cu_q, k_codes, v_codes, k_scale, v_scale, seq_lens, sink,
               window: int | None = None, scale: float | None = None):
    """MTP verify over an 8-bit (E4M3) history: k_codes/v_codes uint8
    [B,Lmax,Hkv,D], k_scale/v_scale [Hkv]; the cache holds code * scale of
    its kv head, so the result is ``verify`` on that dequantized history
    (rounded to fp32, ~6e-8 relative, for the C oracle)."""
    k_codes, v_codes = np.asarray(k_codes, np.uint8), np.asarray(v_codes, np.uint8)
    ks, vs = _f32(k_scale), _f32(v_scale)
    Hkv = k_codes.shape[2]
    if ks.shape != (Hkv,) or vs.shape != (Hkv,) or v_codes.shape != k_codes.shape:
        raise ValueError("oracle.verify_fp8: inconsistent shapes")
    kd = (fp8.decode(k_codes) * ks.astype(np.float64)[None, None, :, None]).astype(np.float32)
    vd = (fp8.decode(v_codes) * vs.astype(np.float64)[None, None, :, None]).astype(np.float32)
    return verify(q, cu_q, kd, vd, seq_lens, sink, window, scale)
