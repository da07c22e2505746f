"""attn_ga_sink_verify_noalloc: GA verify for callers that cannot allocate
device memory (its split-KV scratch is a static device array in the library).
Called through the C ABI, it must give the workspace entry point's result on
two calls in a row with different problems (the shared scratch keeps the
previous call's contents, which must not leak into the next result).

This file sorts last so that a run that stops at the first failure has
already run every other test; it needs nothing from earlier tests."""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_bf16_close

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu

Hq, Hkv, D, PAGE, QMAX = 64, 8, 128, 64, 4


def _problem(ctx, q_lens, seed):
    ctx = np.asarray(ctx, np.int32)
    B = len(ctx)
    npages = (ctx + PAGE - 1) // PAGE
    max_pages = int(npages.max()) + 1
    num_pages = int(npages.sum()) + 5
    perm = synth.page_permutation(num_pages, seed)
    pt = np.zeros((B, max_pages), np.int32)
    o = 0
    for b in range(B):
        pt[b, :npages[b]] = perm[o:o + npages[b]]
        o += npages[b]
    cu_q = synth.cu_seqlens(q_lens)
    return dict(
        q=synth.normal((int(cu_q[-1]), Hq, D), seed + 1, device="cuda"),
        cu_q=torch.from_numpy(cu_q).cuda(),
        kp=synth.normal((num_pages, Hkv, PAGE, D), seed + 2, device="cuda"),
        vp=synth.normal((num_pages, Hkv, PAGE, D), seed + 3, device="cuda"),
        pt=torch.from_numpy(pt).cuda(), ctx=torch.from_numpy(ctx).cuda(),
        sink=synth.sink_logits(Hq, seed + 4, device="cuda"), max_ctx=int(ctx.max()) + 100)


def _call_noalloc(P, out):
    """Raw C-ABI call (ctypes), no Python-side allocation."""
    P_, Hkv_, page_size, _ = P["kp"].shape
    B, max_pages = P["pt"].shape
    vp = ctypes.c_void_p
    st = A._lib.attn_ga_sink_verify_noalloc(
        vp(P["q"].data_ptr()), vp(P["cu_q"].data_ptr()), vp(P["kp"].data_ptr()),
        vp(P["vp"].data_ptr()), vp(P["pt"].data_ptr()), max_pages, P_, page_size,
        vp(P["ctx"].data_ptr()), vp(P["sink"].data_ptr()), vp(out.data_ptr()), B, Hq, Hkv_, D,
        QMAX, P["max_ctx"], ctypes.c_float(1.0 / math.sqrt(D)), A.ATTN_BF16,
        vp(torch.cuda.current_stream().cuda_stream))
    return st


def _history(P, b, L):
    """Request b's first L cached keys and values by position [1, L, Hkv, D],
    gathered from its pages with torch indexing (not this library)."""
    idx = P["pt"][b, :(L + PAGE - 1) // PAGE].long()
    k = P["kp"][idx].transpose(1, 2).reshape(-1, Hkv, D)[:L]
    v = P["vp"][idx].transpose(1, 2).reshape(-1, Hkv, D)[:L]
    return k.cpu()[None], v.cpu()[None]


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    """The larger problem runs first, so split units it left in the shared
    scratch beyond what the second call uses would show in a wrong result.
    Both entry points run the same kernels with the same split layout, so
    their outputs must agree bit for bit; each is also held to the oracle on
    sampled requests."""
    problems = [([300, 9000, 4097, 12000, 20000], [4, 4, 1, 3, 2], 7),
                ([5000, 64, 17000], [2, 4, 4], 8)]
    for ctx, q_lens, seed in problems:
        P = _problem(ctx, np.asarray(q_lens, np.int32), seed)
        assert A.attn_ga_sink_verify_workspace(len(ctx), Hq, Hkv, D, QMAX, P["max_ctx"]) > 0
        ref = A.attn_ga_sink_verify(P["q"], P["cu_q"], P["kp"], P["vp"], P["pt"], P["ctx"],
                                    P["sink"], max_ctx=P["max_ctx"], q_max=QMAX)
        out = torch.full_like(P["q"], float("nan"))
        st = _call_noalloc(P, out)
        assert st == A.ATTN_OK, A._lib.attn_last_error()
        assert A.attn_check_device_error() == 0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"noalloc differs from the workspace entry point (seed {seed})"
        cu = P["cu_q"].cpu().numpy()
        for b in (0, len(ctx) - 1):
            L = int(ctx[b])
            kh, vh = _history(P, b, L)
            r0, r1 = int(cu[b]), int(cu[b + 1])
            r = oracle.verify(P["q"][r0:r1].cpu(), np.array([0, r1 - r0], np.int32), kh, vh,
                              np.array([L], np.int32), P["sink"].cpu(), None)
            assert_bf16_close(out[r0:r1], r, f"noalloc vs oracle (seed {seed}, request {b})")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 64 requests x 8 kv heads x 16 splits of 4096 needs ~136 MB > 64 MiB
    P = _problem([100] * 64, np.full(64, 1, np.int32), 9)
    P["max_ctx"] = 65536
    out = torch.empty_like(P["q"])
    st = _call_noalloc(P, out)
    assert st == A.ATTN_ERR_UNSUPPORTED
    assert b"static scratch" in A._lib.attn_last_error()
