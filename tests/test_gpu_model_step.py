"""One MTP verify step over the whole 48-layer hybrid stack, in model order
(technical-report summary, section "MiMo-V2-Flash Model Architecture": GA at
layers 0, 5, 11, .., 47, SWA elsewhere), captured as one CUDA graph in which
every kernel is a programmatic dependent of the one before it: per layer, the
cache append then the verify.  Each layer's output, read after one replay,
matches the oracle for sampled requests, with that layer's cache (including
the tokens the graph appended) read back by position."""
import numpy as np
import pytest
import torch

import bench
import oracle
from helpers import assert_bf16_close

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu

R, PAGE, W, HKV, D = bench.RING, bench.PAGE, bench.W, bench.HKV, bench.D


def _ring_history(rk, b, L):
    """Ring of request b read out in position order: positions L-n..L-1
    (n = min(L, R)), re-based to 0..n-1, which keeps every query-key distance."""
    n = min(L, R)
    slots = torch.tensor([(L - n + j) % R for j in range(n)], device=rk.device)
    return rk[b][:, slots].transpose(0, 1).cpu()[None], n


def _page_history(pool, pt, b, L):
    idx = pt[b, :(L + PAGE - 1) // PAGE].long()
    return pool[idx].transpose(1, 2).reshape(-1, HKV, D)[:L].cpu()[None]


def test_model_ordered_step_graph_matches_oracle():
    nreq = 5
    q_lens = np.array([4, 1, 4, 3, 2], np.int32)
    ctx = np.array([100, 2600, 700, 131, 1500], np.int32)   # unwrapped, wrapped and full rings
    P = bench.model_step_problem(A, nreq, 0, 0, 77, q_lens=q_lens, ctx=ctx)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bench.model_step(A, P, s)   # eager pass (appends are idempotent)
        torch.cuda.synchronize()
        for d in P["layers"]:
            d["out"].fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            bench.model_step(A, P, s)
        g.replay()
    torch.cuda.synchronize()
    assert A.attn_check_device_error() == 0
    ctx, cu = P["ctx"], P["cu_q_np"]
    sample = [0, 1]   # a ring that has not wrapped, one that has
    for li, d in enumerate(P["layers"]):
        assert torch.isfinite(d["out"].float()).all(), f"layer {li}: rows left unwritten"
        for b in sample:
            L, r0, r1 = int(ctx[b]), int(cu[b]), int(cu[b + 1])
            if d["kind"] == "swa":
                kh, n = _ring_history(d["rk"], b, L)
                vh, _ = _ring_history(d["rv"], b, L)
                window = W
            else:
                kh, vh, n = _page_history(d["kp"], d["pt"], b, L), _page_history(d["vp"], d["pt"], b, L), L
                window = None
            # the appended tokens are the cache's last q_len positions
            assert torch.equal(kh[0, n - (r1 - r0):], d["k_new"][r0:r1].cpu())
            ref = oracle.verify(d["q"][r0:r1].cpu(), np.array([0, r1 - r0], np.int32), kh, vh,
                                np.array([n], np.int32), d["sink"].cpu(), window)
            assert_bf16_close(d["out"][r0:r1], ref, f"layer {li} ({d['kind']}) request {b}")
