"""Thin Python binding of ``libattn_sink.so`` (B300 / sm_103a sink attention).

Each function has the name of the C entry point it wraps (see
``include/attn_sink.h``) and only marshals arguments: it checks shapes, dtypes
and devices of torch tensors, passes their device pointers and sizes through
ctypes, and enqueues on the current CUDA stream.  All computation happens in
the library's CUDA kernels; there is no fallback, and importing this package
fails when the library has not been built.

The operation: causal attention over a sliding window of W keys (SWA) or the
full prefix (GA) with one learnable sink logit per query head that joins the
softmax denominator and carries no value (MiMo-V2-Flash technical-report
summary, sections "MiMo-V2-Flash Model Architecture" and "Hybrid Sliding
Window Attention Architecture"), in prefill and in the MTP verify step
(release announcement "小米开源 MiMo-V2-Flash", figure "Multi-Token Prediction").
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn_sink.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "attn_sink.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m global_attention_sinks_swa_b300._build` "
        "(this package has no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_FAULT = range(5)
ATTN_BF16, ATTN_F32 = 0, 1
DEVERR_PAGE_OOB, DEVERR_CTX_OOB, DEVERR_QLEN, DEVERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4, 0x8
DEVERR_SEQLENS = 0x10

_vp, _ci, _cf, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "attn_version": ([], _ci),
    "attn_last_error": ([], ctypes.c_char_p),
    "attn_check_device_error": ([_vp, ctypes.POINTER(ctypes.c_uint)], _ci),
    "attn_swa_sink_prefill": ([_vp] * 6 + [_ci] * 6 + [_cf, _ci, _vp], _ci),
    "attn_ga_sink_prefill": ([_vp] * 6 + [_ci] * 5 + [_cf, _ci, _vp], _ci),
    "attn_sink_prefill_backward_workspace": ([_ci] * 4, _sz),
    "attn_sink_prefill_backward": ([_vp] * 12 + [_sz] + [_ci] * 6 + [_cf, _ci, _vp], _ci),
    "attn_swa_sink_prefill_varlen": ([_vp] * 7 + [_ci] * 7 + [_cf, _cf, _ci, _vp], _ci),
    "attn_ga_sink_prefill_varlen": ([_vp] * 7 + [_ci] * 6 + [_cf, _cf, _ci, _vp], _ci),
    "attn_swa_ring_append": ([_vp] * 6 + [_ci] * 6 + [_vp], _ci),
    "attn_ga_paged_append": ([_vp] * 7 + [_ci] * 8 + [_vp], _ci),
    "attn_swa_sink_verify": ([_vp] * 7 + [_ci] * 7 + [_cf, _ci, _vp], _ci),
    "attn_ga_sink_verify_workspace": ([_ci] * 6, _sz),
    "attn_ga_sink_verify": ([_vp] * 5 + [_ci] * 3 + [_vp] * 4 + [_sz] + [_ci] * 6 + [_cf, _ci, _vp], _ci),
    "attn_ga_paged_append_fp8": ([_vp] * 7 + [_ci] * 3 + [_vp, _vp] + [_ci] * 4 + [_vp], _ci),
    "attn_ga_sink_verify_fp8": ([_vp] * 5 + [_ci] * 3 + [_vp] * 6 + [_sz] + [_ci] * 6 + [_cf, _vp], _ci),
    "attn_ga_sink_verify_noalloc": ([_vp] * 5 + [_ci] * 3 + [_vp] * 3 + [_ci] * 6 + [_cf, _ci, _vp], _ci),
    "attn_debug_prefill_visits": ([_vp] + [_ci] * 4 + [_vp], _ci),
    "attn_debug_swa_stream_visits": ([_vp] + [_ci] * 5 + [_vp], _ci),
    "attn_debug_verify_positions": ([_vp, _ci, _vp, _vp] + [_ci] * 6 + [_vp], _ci),
    "attn_debug_wait_timeout": ([_vp], _ci),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class AttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"attn status {status}: {msg}")
        self.status = status


def declared_symbols() -> list[str]:
    """Names of the functions declared in include/attn_sink.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:[A-Za-z_][\w\s\*]*?)\b(attn_\w+)\s*\(", text, re.M)))


def _check(status: int):
    if status != ATTN_OK:
        raise AttnError(status, (_lib.attn_last_error() or b"").decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _expect(t, shape, dtype, what):
    """The library trusts the sizes it is given: every buffer must match them."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape) or (dtype is not None and t.dtype != dtype):
        raise ValueError(f"{what} must be {dtype} {list(shape)}, got {t.dtype} {list(t.shape)}")


def attn_version() -> int:
    return _lib.attn_version()


def attn_check_device_error(stream=None) -> int:
    """Synchronise `stream` and return (and clear) the device error bits."""
    bits = ctypes.c_uint(0)
    st = _lib.attn_check_device_error(_stream(stream), ctypes.byref(bits))
    if st not in (ATTN_OK, ATTN_ERR_DEVICE_FAULT):
        _check(st)
    return bits.value


def _prefill(swa: bool, q, k, v, sink, window, scale, out, lse, stream):
    _cuda(q, k, v, sink, out, lse)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, T, Hkv, D) or v.shape != k.shape or sink.shape != (Hq,):
        raise ValueError("shapes: q [B,T,Hq,D], k/v [B,T,Hkv,D], sink [Hq]")
    if k.dtype != q.dtype or v.dtype != q.dtype or sink.dtype != torch.float32:
        raise TypeError("q/k/v share one dtype; sink is float32")
    _expect(out, q.shape, q.dtype, "out")
    out = torch.empty_like(q) if out is None else out
    if lse is not None and (lse.shape != (B, Hq, T) or lse.dtype != torch.float32):
        raise ValueError("lse must be float32 [B,Hq,T]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(sink), _ptr(out), _ptr(lse), B, T, Hq, Hkv, D]
    if swa:
        st = _lib.attn_swa_sink_prefill(*args, int(window), scale, _dtype_code(q), _stream(stream))
    else:
        st = _lib.attn_ga_sink_prefill(*args, scale, _dtype_code(q), _stream(stream))
    _check(st)
    return out


def attn_swa_sink_prefill(q, k, v, sink, window: int = 128, scale: float | None = None,
                          out=None, lse=None, stream=None):
    """Sliding-window sink attention over whole sequences.
    q [B,T,Hq,D], k/v [B,T,Hkv,D] (bf16 or fp32), sink [Hq] fp32 -> o [B,T,Hq,D]."""
    return _prefill(True, q, k, v, sink, window, scale, out, lse, stream)


def attn_ga_sink_prefill(q, k, v, sink, scale: float | None = None, out=None, lse=None,
                         stream=None):
    """Global (full causal) sink attention over whole sequences."""
    return _prefill(False, q, k, v, sink, 0, scale, out, lse, stream)


def _prefill_varlen(swa: bool, q, k, v, cu_seqlens, sink, window, max_seqlen, scale,
                    value_scale, out, lse, stream):
    _cuda(q, k, v, cu_seqlens, sink, out, lse)
    total, Hq, D = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.shape[0] - 1
    if k.shape != (total, Hkv, D) or v.shape != k.shape or sink.shape != (Hq,) or B < 0:
        raise ValueError("shapes: q [total,Hq,D], k/v [total,Hkv,D], cu_seqlens [B+1], sink [Hq]")
    if k.dtype != q.dtype or v.dtype != q.dtype or sink.dtype != torch.float32:
        raise TypeError("q/k/v share one dtype; sink is float32")
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens is int32")
    if max_seqlen is None:  # one device-to-host read; pass it to stay asynchronous
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if B > 0 else 0
    _expect(out, q.shape, q.dtype, "out")
    out = torch.empty_like(q) if out is None else out
    if lse is not None and (lse.shape != (Hq, total) or lse.dtype != torch.float32):
        raise ValueError("lse must be float32 [Hq,total]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(sink), _ptr(out), _ptr(lse), B,
            total, int(max_seqlen), Hq, Hkv, D]
    if swa:
        st = _lib.attn_swa_sink_prefill_varlen(*args, int(window), scale, float(value_scale),
                                               _dtype_code(q), _stream(stream))
    else:
        st = _lib.attn_ga_sink_prefill_varlen(*args, scale, float(value_scale), _dtype_code(q),
                                              _stream(stream))
    _check(st)
    return out


def attn_swa_sink_prefill_varlen(q, k, v, cu_seqlens, sink, window: int = 128,
                                 max_seqlen: int | None = None, scale: float | None = None,
                                 value_scale: float = 1.0, out=None, lse=None, stream=None):
    """Sliding-window sink attention over a packed batch of sequences.
    q [total,Hq,D], k/v [total,Hkv,D], cu_seqlens [B+1] int32 (device),
    sink [Hq] fp32 -> o [total,Hq,D] = value_scale * attention; lse [Hq,total]."""
    return _prefill_varlen(True, q, k, v, cu_seqlens, sink, window, max_seqlen, scale,
                           value_scale, out, lse, stream)


def attn_ga_sink_prefill_varlen(q, k, v, cu_seqlens, sink, max_seqlen: int | None = None,
                                scale: float | None = None, value_scale: float = 1.0, out=None,
                                lse=None, stream=None):
    """Global (full causal) sink attention over a packed batch of sequences."""
    return _prefill_varlen(False, q, k, v, cu_seqlens, sink, 0, max_seqlen, scale, value_scale,
                           out, lse, stream)


def attn_sink_prefill_backward(q, k, v, o, lse, dout, sink, window: int = 0,
                               scale: float | None = None, workspace=None, stream=None):
    """Gradients of the bf16 prefill: returns (dq, dk, dv, dsink).  o and lse
    [B,Hq,T] come from the forward call (window 0 = global attention)."""
    _cuda(q, k, v, o, lse, dout, sink, workspace)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if o.shape != q.shape or dout.shape != q.shape or lse.shape != (B, Hq, T):
        raise ValueError("o/dout [B,T,Hq,D] and lse [B,Hq,T] must match q")
    for t, name in ((k, "k"), (v, "v")):
        _expect(t, (B, T, Hkv, D), q.dtype, name)
    for t, name in ((o, "o"), (dout, "dout")):
        _expect(t, q.shape, q.dtype, name)
    _expect(lse, (B, Hq, T), torch.float32, "lse")
    _expect(sink, (Hq,), torch.float32, "sink")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsink = torch.empty(Hq, dtype=torch.float32, device=q.device)
    need = _lib.attn_sink_prefill_backward_workspace(B, T, Hq, D)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(_lib.attn_sink_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                           _ptr(dout), _ptr(sink), _ptr(dq), _ptr(dk), _ptr(dv),
                                           _ptr(dsink), _ptr(workspace), ws_bytes, B, T, Hq, Hkv,
                                           D, int(window), scale, _dtype_code(q),
                                           _stream(stream)))
    return dq, dk, dv, dsink


def _append_common(k_new, v_new, cu_q, seq_lens, kc, vc):
    _cuda(k_new, v_new, cu_q, seq_lens, kc, vc)
    if cu_q.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("cu_q and seq_lens are int32")
    if k_new.dtype != kc.dtype or v_new.dtype != vc.dtype or k_new.shape != v_new.shape:
        raise TypeError("new keys/values must match the cache dtype and each other")
    if k_new.dim() != 3 or seq_lens.dim() != 1:
        raise ValueError("k_new/v_new [rows,Hkv,D], seq_lens [B]")
    _expect(cu_q, (seq_lens.shape[0] + 1,), torch.int32, "cu_q")
    return seq_lens.shape[0], k_new.shape[1], k_new.shape[2]


def attn_swa_ring_append(k_new, v_new, cu_q, seq_lens, ring_k, ring_v, q_max: int, stream=None):
    """Write each request's new keys/values into slot p mod R of its ring
    (ring_k/ring_v [B,Hkv,R,D]); seq_lens counts the new tokens."""
    B, Hkv, D = _append_common(k_new, v_new, cu_q, seq_lens, ring_k, ring_v)
    if ring_k.shape[:2] != (B, Hkv) or ring_k.shape[3] != D or ring_v.shape != ring_k.shape:
        raise ValueError("ring_k/ring_v must be [B,Hkv,R,D]")
    _check(_lib.attn_swa_ring_append(_ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(seq_lens),
                                     _ptr(ring_k), _ptr(ring_v), B, Hkv, D, ring_k.shape[2],
                                     int(q_max), _dtype_code(k_new), _stream(stream)))


def attn_ga_paged_append(k_new, v_new, cu_q, seq_lens, k_pages, v_pages, page_table, q_max: int,
                         stream=None):
    """Write each request's new keys/values into its pages
    (k_pages/v_pages [P,Hkv,page,D], page_table [B,max_pages] int32)."""
    B, Hkv, D = _append_common(k_new, v_new, cu_q, seq_lens, k_pages, v_pages)
    _cuda(page_table)
    if page_table.dtype != torch.int32 or page_table.shape[0] != B:
        raise ValueError("page_table must be int32 [B,max_pages]")
    if k_pages.shape[1] != Hkv or k_pages.shape[3] != D or v_pages.shape != k_pages.shape:
        raise ValueError("k_pages/v_pages must be [P,Hkv,page_size,D]")
    _check(_lib.attn_ga_paged_append(_ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(seq_lens),
                                     _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                     page_table.shape[1], k_pages.shape[0], k_pages.shape[2], B,
                                     Hkv, D, int(q_max), _dtype_code(k_new), _stream(stream)))


def attn_swa_sink_verify(q, cu_q, ring_k, ring_v, seq_lens, sink, window: int = 128,
                         q_max: int = 4, scale: float | None = None, out=None, stream=None):
    """MTP verify against the SWA ring.  q [sum_q,Hq,D] bf16 -> o [sum_q,Hq,D]."""
    _cuda(q, cu_q, ring_k, ring_v, seq_lens, sink, out)
    nq, Hq, D = q.shape
    B, Hkv, R, _ = ring_k.shape
    if cu_q.shape != (B + 1,) or seq_lens.shape != (B,) or sink.shape != (Hq,):
        raise ValueError("cu_q [B+1], seq_lens [B], sink [Hq]")
    _expect(ring_k, (B, Hkv, R, D), q.dtype, "ring_k")
    _expect(ring_v, (B, Hkv, R, D), q.dtype, "ring_v")
    _expect(cu_q, (B + 1,), torch.int32, "cu_q")
    _expect(seq_lens, (B,), torch.int32, "seq_lens")
    _expect(sink, (Hq,), torch.float32, "sink")
    _expect(out, q.shape, q.dtype, "out")
    out = torch.empty_like(q) if out is None else out
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(_lib.attn_swa_sink_verify(_ptr(q), _ptr(cu_q), _ptr(ring_k), _ptr(ring_v),
                                     _ptr(seq_lens), _ptr(sink), _ptr(out), B, Hq, Hkv, D,
                                     int(window), R, int(q_max), scale, _dtype_code(q),
                                     _stream(stream)))
    return out


def attn_ga_sink_verify_workspace(B: int, Hq: int, Hkv: int, D: int, q_max: int,
                                  max_ctx: int) -> int:
    return int(_lib.attn_ga_sink_verify_workspace(B, Hq, Hkv, D, q_max, max_ctx))


def _paged_checks(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, out, page_dtype):
    nq, Hq, D = q.shape
    P, Hkv, page_size, _ = k_pages.shape
    B, max_pages = page_table.shape
    _expect(k_pages, (P, Hkv, page_size, D), page_dtype, "k_pages")
    _expect(v_pages, (P, Hkv, page_size, D), page_dtype, "v_pages")
    _expect(page_table, (B, max_pages), torch.int32, "page_table")
    _expect(cu_q, (B + 1,), torch.int32, "cu_q")
    _expect(seq_lens, (B,), torch.int32, "seq_lens")
    _expect(sink, (Hq,), torch.float32, "sink")
    _expect(out, q.shape, q.dtype, "out")
    return nq, Hq, D, P, Hkv, page_size, B, max_pages


def attn_ga_sink_verify(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, max_ctx: int,
                        q_max: int = 4, scale: float | None = None, out=None, workspace=None,
                        stream=None):
    """MTP verify against the GA paged cache (split-KV + LSE merge)."""
    _cuda(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, out, workspace)
    nq, Hq, D, P, Hkv, page_size, B, max_pages = _paged_checks(
        q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, out, q.dtype)
    out = torch.empty_like(q) if out is None else out
    need = attn_ga_sink_verify_workspace(B, Hq, Hkv, D, q_max, max_ctx)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(_lib.attn_ga_sink_verify(_ptr(q), _ptr(cu_q), _ptr(k_pages), _ptr(v_pages),
                                    _ptr(page_table), max_pages, P, page_size, _ptr(seq_lens),
                                    _ptr(sink), _ptr(out), _ptr(workspace), ws_bytes, B, Hq, Hkv,
                                    D, int(q_max), int(max_ctx), scale, _dtype_code(q),
                                    _stream(stream)))
    return out


def attn_ga_sink_verify_fp8(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, k_scale,
                            v_scale, max_ctx: int, q_max: int = 4, scale: float | None = None,
                            out=None, workspace=None, stream=None):
    """MTP verify against an 8-bit (E4M3) GA paged cache: k_pages/v_pages uint8
    [P,Hkv,page,D] codes, entry = code * k_scale[g] (v_scale[g]); q/o bf16."""
    _cuda(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, k_scale, v_scale, out, workspace)
    if k_pages.dtype != torch.uint8 or v_pages.dtype != torch.uint8:
        raise TypeError("8-bit pages are uint8 E4M3 codes")
    if k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32:
        raise TypeError("k_scale/v_scale are float32 [Hkv]")
    nq, Hq, D, P, Hkv, page_size, B, max_pages = _paged_checks(
        q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, out, torch.uint8)
    _expect(k_scale, (Hkv,), torch.float32, "k_scale")
    _expect(v_scale, (Hkv,), torch.float32, "v_scale")
    out = torch.empty_like(q) if out is None else out
    need = attn_ga_sink_verify_workspace(B, Hq, Hkv, D, q_max, max_ctx)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(_lib.attn_ga_sink_verify_fp8(_ptr(q), _ptr(cu_q), _ptr(k_pages), _ptr(v_pages),
                                        _ptr(page_table), max_pages, P, page_size, _ptr(seq_lens),
                                        _ptr(sink), _ptr(k_scale), _ptr(v_scale), _ptr(out),
                                        _ptr(workspace), ws_bytes, B, Hq, Hkv, D, int(q_max),
                                        int(max_ctx), scale, _stream(stream)))
    return out


def attn_ga_paged_append_fp8(k_new, v_new, cu_q, seq_lens, k_pages, v_pages, page_table,
                             k_scale, v_scale, q_max: int, stream=None):
    """Quantize each request's new bf16 keys/values to E4M3 codes of
    value / scale[kv head] and write them into its 8-bit pages."""
    _cuda(k_new, v_new, cu_q, seq_lens, k_pages, v_pages, page_table, k_scale, v_scale)
    if k_new.dtype != torch.bfloat16 or v_new.dtype != torch.bfloat16 or k_new.shape != v_new.shape:
        raise TypeError("new keys/values are bf16 [rows,Hkv,D]")
    if k_pages.dtype != torch.uint8 or v_pages.shape != k_pages.shape:
        raise TypeError("8-bit pages are uint8 [P,Hkv,page,D]")
    if cu_q.dtype != torch.int32 or seq_lens.dtype != torch.int32 or page_table.dtype != torch.int32:
        raise TypeError("cu_q, seq_lens and page_table are int32")
    B = seq_lens.shape[0]
    Hkv, D = k_new.shape[1], k_new.shape[2]
    if k_new.dim() != 3 or k_pages.dim() != 4 or k_pages.shape[1] != Hkv or k_pages.shape[3] != D:
        raise ValueError("k_new/v_new [rows,Hkv,D], k_pages/v_pages [P,Hkv,page,D]")
    if page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("page_table must be int32 [B,max_pages]")
    _expect(cu_q, (B + 1,), torch.int32, "cu_q")
    _expect(k_scale, (Hkv,), torch.float32, "k_scale")
    _expect(v_scale, (Hkv,), torch.float32, "v_scale")
    _check(_lib.attn_ga_paged_append_fp8(_ptr(k_new), _ptr(v_new), _ptr(cu_q), _ptr(seq_lens),
                                         _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
                                         page_table.shape[1], k_pages.shape[0], k_pages.shape[2],
                                         _ptr(k_scale), _ptr(v_scale), B, Hkv, D, int(q_max),
                                         _stream(stream)))


def attn_ga_sink_verify_noalloc(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink,
                                max_ctx: int, q_max: int = 4, scale: float | None = None,
                                out=None, stream=None):
    """attn_ga_sink_verify for callers that cannot allocate device memory: the
    split-KV scratch is the library's static 64 MiB device array (see the C
    header for its limits; concurrent calls on one device race on it)."""
    _cuda(q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, out)
    nq, Hq, D, P, Hkv, page_size, B, max_pages = _paged_checks(
        q, cu_q, k_pages, v_pages, page_table, seq_lens, sink, out, q.dtype)
    if out is None:
        raise ValueError("pass a preallocated `out` (this entry point allocates nothing)")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(_lib.attn_ga_sink_verify_noalloc(_ptr(q), _ptr(cu_q), _ptr(k_pages), _ptr(v_pages),
                                            _ptr(page_table), max_pages, P, page_size,
                                            _ptr(seq_lens), _ptr(sink), _ptr(out), B, Hq, Hkv, D,
                                            int(q_max), int(max_ctx), scale, _dtype_code(q),
                                            _stream(stream)))
    return out


def attn_debug_prefill_visits(T: int, window: int, mode: int, G: int = 8, device="cuda",
                              stream=None):
    """[T,T] int32 visit counts of the prefill tiling (mode 0 GA tiles, 1 packed SWA)."""
    visits = torch.empty(T, T, dtype=torch.int32, device=device)
    _check(_lib.attn_debug_prefill_visits(_ptr(visits), int(mode), T, int(window), int(G),
                                          _stream(stream)))
    return visits


def attn_debug_swa_stream_visits(B: int, T: int, Hkv: int, window: int = 128, grid: int = 0,
                                 device="cuda", stream=None):
    """[B*Hkv,T,T+1] int32 visit counts of the streaming SWA prefill schedule
    (column T counts admitted keys outside [0,T)); grid 0 = the kernel's own."""
    visits = torch.zeros(B * Hkv, T, T + 1, dtype=torch.int32, device=device)
    _check(_lib.attn_debug_swa_stream_visits(_ptr(visits), B, T, Hkv, int(window), int(grid),
                                             _stream(stream)))
    return visits


def attn_debug_verify_positions(kind: int, cu_q, seq_lens, q_max: int, window: int,
                                ring_slots: int = 0, max_pages: int = 0, page_size: int = 64,
                                stream=None):
    """Positions the verify kernels assign to cache slots (see the C header)."""
    _cuda(cu_q, seq_lens)
    B = seq_lens.shape[0]
    n = ring_slots if kind == 0 else max_pages * page_size
    out = torch.empty(B, q_max, n, dtype=torch.int32, device=seq_lens.device)
    _check(_lib.attn_debug_verify_positions(_ptr(out), int(kind), _ptr(cu_q), _ptr(seq_lens), B,
                                            int(q_max), int(window), int(ring_slots),
                                            int(max_pages), int(page_size), _stream(stream)))
    return out


def attn_debug_wait_timeout(stream=None):
    """Enqueue a kernel whose pipeline wait runs out (about 2 s) and sets
    DEVERR_WAIT_TIMEOUT; read and clear it with attn_check_device_error()."""
    _check(_lib.attn_debug_wait_timeout(_stream(stream)))
