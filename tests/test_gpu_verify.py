"""MTP verify parity: the CUDA verify kernels (SWA ring, GA paged with
split-KV) and the KV appends, through the C ABI, against the fp64 oracle that
reads keys/values by position from a linear history."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_bf16_close
from oracle import index

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu

Hq, Hkv, D, W, QMAX, PAGE = 64, 8, 128, 128, 4, 64
R = index.ring_slots(W, QMAX)


def ring_from_history(k_hist, seq_lens, slots=R):
    """[B,Lmax,Hkv,D] -> ring [B,Hkv,slots,D] holding positions max(0,L-slots)..L-1."""
    B, _, hkv, _ = k_hist.shape
    ring = torch.zeros(B, hkv, slots, D, dtype=k_hist.dtype)
    for b in range(B):
        L = int(seq_lens[b])
        for p in range(max(0, L - slots), L):
            ring[b, :, index.ring_slot(p, slots)] = k_hist[b, p]
    return ring


def pages_from_history(k_hist, seq_lens, page_table, num_pages):
    B = k_hist.shape[0]
    pool = torch.zeros(num_pages, Hkv, PAGE, D, dtype=k_hist.dtype)
    for b in range(B):
        L = int(seq_lens[b])
        for p0 in range(0, L, PAGE):
            n = min(PAGE, L - p0)
            page, off = index.page_location(page_table, b, p0, PAGE)
            pool[page, :, off:off + n] = k_hist[b, p0:p0 + n].transpose(0, 1)
    return pool


def make_problem(seq_lens, q_lens, seed, extra_pages=3):
    seq_lens = np.asarray(seq_lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    B, Lmax = len(seq_lens), int(seq_lens.max())
    k_hist = synth.normal((B, Lmax, Hkv, D), seed)
    v_hist = synth.normal((B, Lmax, Hkv, D), seed + 1)
    cu_q = synth.cu_seqlens(q_lens)
    q = synth.normal((int(cu_q[-1]), Hq, D), seed + 2)
    sink = synth.sink_logits(Hq, seed + 3)
    max_pages = (Lmax + PAGE - 1) // PAGE
    num_pages = B * max_pages + extra_pages
    perm = synth.page_permutation(num_pages, seed + 4)
    page_table = perm[:B * max_pages].reshape(B, max_pages).copy()
    return dict(seq_lens=seq_lens, q_lens=q_lens, k_hist=k_hist, v_hist=v_hist, cu_q=cu_q, q=q,
                sink=sink, page_table=page_table, num_pages=num_pages, Lmax=Lmax)


def run_ring(P, sink=None):
    sink = P["sink"] if sink is None else sink
    rk = ring_from_history(P["k_hist"], P["seq_lens"]).cuda()
    rv = ring_from_history(P["v_hist"], P["seq_lens"]).cuda()
    o = A.attn_swa_sink_verify(P["q"].cuda(), torch.from_numpy(P["cu_q"]).cuda(), rk, rv,
                               torch.from_numpy(P["seq_lens"]).cuda(), sink.cuda(), window=W,
                               q_max=QMAX)
    assert A.attn_check_device_error() == 0
    return o


def run_paged(P, max_ctx=None, sink=None):
    sink = P["sink"] if sink is None else sink
    kp = pages_from_history(P["k_hist"], P["seq_lens"], P["page_table"], P["num_pages"]).cuda()
    vp = pages_from_history(P["v_hist"], P["seq_lens"], P["page_table"], P["num_pages"]).cuda()
    max_ctx = int(P["seq_lens"].max()) if max_ctx is None else max_ctx
    o = A.attn_ga_sink_verify(P["q"].cuda(), torch.from_numpy(P["cu_q"]).cuda(), kp, vp,
                              torch.from_numpy(P["page_table"]).cuda(),
                              torch.from_numpy(P["seq_lens"]).cuda(), sink.cuda(), max_ctx=max_ctx,
                              q_max=QMAX)
    assert A.attn_check_device_error() == 0
    return o


def ref(P, window, sink=None):
    sink = P["sink"] if sink is None else sink
    return oracle.verify(P["q"], P["cu_q"], P["k_hist"], P["v_hist"], P["seq_lens"], sink, window)


CASES = [
    ([4, 50, 131, 132, 700], [4, 1, 3, 4, 2]),
    ([1, 2, 3, 4], [1, 2, 3, 4]),
    ([129, 130, 131, 260, 261, 262, 263, 5000], [4, 4, 4, 4, 3, 2, 1, 4]),
]


@pytest.mark.parametrize("seq_lens,q_lens", CASES)
def test_swa_ring_verify(seq_lens, q_lens):
    P = make_problem(seq_lens, q_lens, seed=sum(seq_lens))
    assert_bf16_close(run_ring(P), ref(P, W), "ring verify")


@pytest.mark.parametrize("window,hq,hkv", [
    (8, 64, 8),     # tensor-core kernel, ring of 11 slots
    (141, 64, 8),   # tensor-core kernel, ring of 144 slots (its largest)
    (200, 64, 8),   # ring of 203 slots: mma.sync kernel
    (128, 32, 8),   # 4 q-heads per kv head: mma.sync kernel
    (5, 16, 4),     # 4 q-heads per kv head, small window
])
def test_swa_ring_verify_both_kernels(window, hq, hkv):
    """The ring verify on both of its kernels (tcgen05 for 8 q-heads per kv head
    and rings <= 144 slots, mma.sync otherwise) against the oracle."""
    seq_lens = np.array([3, 9, 150, 151, 260, 1000], np.int32)
    q_lens = np.array([3, 4, 4, 1, 2, 4], np.int32)
    B, Lmax = len(seq_lens), int(seq_lens.max())
    seed = window + hq
    k_hist = synth.normal((B, Lmax, hkv, D), seed)
    v_hist = synth.normal((B, Lmax, hkv, D), seed + 1)
    cu_q = synth.cu_seqlens(q_lens)
    q = synth.normal((int(cu_q[-1]), hq, D), seed + 2)
    sink = synth.sink_logits(hq, seed + 3)
    R = index.ring_slots(window, QMAX)
    rk = ring_from_history(k_hist, seq_lens, R).cuda()
    rv = ring_from_history(v_hist, seq_lens, R).cuda()
    o = A.attn_swa_sink_verify(q.cuda(), torch.from_numpy(cu_q).cuda(), rk, rv,
                               torch.from_numpy(seq_lens).cuda(), sink.cuda(), window=window,
                               q_max=QMAX)
    assert A.attn_check_device_error() == 0
    ref_o = oracle.verify(q, cu_q, k_hist, v_hist, seq_lens, sink, window)
    assert_bf16_close(o, ref_o, f"ring verify W={window} G={hq // hkv}")


@pytest.mark.parametrize("seq_lens,q_lens", CASES + [([4097, 9000, 64, 65], [4, 3, 1, 4])])
def test_ga_paged_verify(seq_lens, q_lens):
    P = make_problem(seq_lens, q_lens, seed=3 * sum(seq_lens))
    assert_bf16_close(run_paged(P), ref(P, None), "paged verify")


def test_ga_paged_verify_split_paths_agree():
    """One split (max_ctx <= 4096, merged in-kernel) and many splits (combine
    kernel) give the oracle's result for the same problem."""
    P = make_problem([300, 4000, 1000], [4, 4, 2], seed=11)
    r = ref(P, None)
    assert_bf16_close(run_paged(P, max_ctx=4096), r, "1 split")
    assert_bf16_close(run_paged(P, max_ctx=20000), r, "5 splits")


def test_verify_extreme_sinks():
    P = make_problem([10, 300, 5000], [4, 4, 1], seed=21)
    sink = P["sink"].clone()
    sink[0], sink[7], sink[8], sink[63] = math.inf, -math.inf, 25.0, -25.0
    o = run_ring(P, sink)
    assert_bf16_close(o, ref(P, W, sink), "ring sinks")
    assert torch.all(o[:, 0] == 0)
    o = run_paged(P, sink=sink)
    assert_bf16_close(o, ref(P, None, sink), "paged sinks")
    assert torch.all(o[:, 0] == 0)


def test_appends_bit_exact():
    """Ring and paged appends place every new row where the index
    definitions say, and touch nothing else."""
    seq_lens = np.array([4, 131, 140, 1000], np.int32)
    q_lens = np.array([4, 2, 4, 1], np.int32)
    P = make_problem(seq_lens, q_lens, seed=5)
    cu_q = P["cu_q"]
    k_new = synth.normal((int(cu_q[-1]), Hkv, D), 90)
    v_new = synth.normal((int(cu_q[-1]), Hkv, D), 91)
    B = len(seq_lens)
    ring_k = synth.normal((B, Hkv, R, D), 92).cuda()
    ring_v = synth.normal((B, Hkv, R, D), 93).cuda()
    exp_k, exp_v = ring_k.cpu().clone(), ring_v.cpu().clone()
    kp = synth.normal((P["num_pages"], Hkv, PAGE, D), 94).cuda()
    vp = synth.normal((P["num_pages"], Hkv, PAGE, D), 95).cuda()
    exp_kp, exp_vp = kp.cpu().clone(), vp.cpu().clone()
    for b in range(B):
        for t in range(int(q_lens[b])):
            p = int(seq_lens[b]) - int(q_lens[b]) + t
            exp_k[b, :, index.ring_slot(p, R)] = k_new[cu_q[b] + t]
            exp_v[b, :, index.ring_slot(p, R)] = v_new[cu_q[b] + t]
            page, off = index.page_location(P["page_table"], b, p, PAGE)
            exp_kp[page, :, off] = k_new[cu_q[b] + t]
            exp_vp[page, :, off] = v_new[cu_q[b] + t]
    cu = torch.from_numpy(cu_q).cuda()
    sl = torch.from_numpy(seq_lens).cuda()
    A.attn_swa_ring_append(k_new.cuda(), v_new.cuda(), cu, sl, ring_k, ring_v, q_max=QMAX)
    A.attn_ga_paged_append(k_new.cuda(), v_new.cuda(), cu, sl, kp, vp,
                           torch.from_numpy(P["page_table"]).cuda(), q_max=QMAX)
    assert A.attn_check_device_error() == 0
    assert torch.equal(ring_k.cpu(), exp_k) and torch.equal(ring_v.cpu(), exp_v)
    assert torch.equal(kp.cpu(), exp_kp) and torch.equal(vp.cpu(), exp_vp)


def test_mtp_walk_sequence():
    """A synthetic MTP loop of 200 passes: each pass appends 1 real + up to 3
    draft tokens per request through the append kernels, verifies them against
    the ring and the pages, then accepts a random prefix per request (drawn
    per pass and request) and rolls the length back, so the next append
    overwrites the rejected slots.  Every pass matches the oracle on the
    linear history."""
    B, steps = 3, 200
    L0 = np.array([0, 127, 4090], np.int32)
    Lcap = int(L0.max()) + steps * QMAX + 8
    k_hist = synth.normal((B, Lcap, Hkv, D), 100)
    v_hist = synth.normal((B, Lcap, Hkv, D), 101)
    # fp32 copies (exact) for the oracle, kept in step with the bf16 history
    k32 = k_hist.float().numpy().copy()
    v32 = v_hist.float().numpy().copy()
    sink = synth.sink_logits(Hq, 102)
    max_pages = (Lcap + PAGE - 1) // PAGE
    num_pages = B * max_pages
    page_table = synth.page_permutation(num_pages, 103).reshape(B, max_pages)
    hist0 = np.maximum(L0, 0)
    ring_k = ring_from_history(k_hist, hist0).cuda()
    ring_v = ring_from_history(v_hist, hist0).cuda()
    kp = pages_from_history(k_hist, hist0, page_table, num_pages).cuda()
    vp = pages_from_history(v_hist, hist0, page_table, num_pages).cuda()
    pt = torch.from_numpy(page_table).cuda()
    accepts = synth.accept_counts(steps * B, QMAX, 104).reshape(steps, B)
    sink_d = sink.cuda()
    base = L0.copy()
    for s in range(steps):
        q_lens = np.array([QMAX if (s + b) % 7 else 1 + (s % QMAX) for b in range(B)], np.int32)
        seq_lens = (base + q_lens).astype(np.int32)
        cu_q = synth.cu_seqlens(q_lens)
        # fresh tokens for this pass (a rejected draft gets new values next time)
        k_new = synth.normal((int(cu_q[-1]), Hkv, D), 1000 + s)
        v_new = synth.normal((int(cu_q[-1]), Hkv, D), 2000 + s)
        for b in range(B):
            k32[b, base[b]:seq_lens[b]] = k_new[cu_q[b]:cu_q[b + 1]].float().numpy()
            v32[b, base[b]:seq_lens[b]] = v_new[cu_q[b]:cu_q[b + 1]].float().numpy()
        cu, sl = torch.from_numpy(cu_q).cuda(), torch.from_numpy(seq_lens).cuda()
        A.attn_swa_ring_append(k_new.cuda(), v_new.cuda(), cu, sl, ring_k, ring_v, q_max=QMAX)
        A.attn_ga_paged_append(k_new.cuda(), v_new.cuda(), cu, sl, kp, vp, pt, q_max=QMAX)
        q = synth.normal((int(cu_q[-1]), Hq, D), 3000 + s)
        o_ring = A.attn_swa_sink_verify(q.cuda(), cu, ring_k, ring_v, sl, sink_d, window=W,
                                        q_max=QMAX)
        o_pg = A.attn_ga_sink_verify(q.cuda(), cu, kp, vp, pt, sl, sink_d, max_ctx=Lcap,
                                     q_max=QMAX)
        assert A.attn_check_device_error() == 0
        assert_bf16_close(o_ring, oracle.verify(q, cu_q, k32, v32, seq_lens, sink, W),
                          f"ring step {s}")
        assert_bf16_close(o_pg, oracle.verify(q, cu_q, k32, v32, seq_lens, sink, None),
                          f"paged step {s}")
        base = base + 1 + np.minimum(accepts[s], q_lens - 1)


# ------------------------------------------------------- full sizes, sampled
def _full_problem(ctx, q_lens, seed):
    """Paged pool filled on the device by the seeded generator."""
    ctx = np.asarray(ctx, np.int32)
    B = len(ctx)
    npages = (ctx + PAGE - 1) // PAGE
    max_pages = int(npages.max())
    num_pages = int(npages.sum())
    perm = synth.page_permutation(num_pages, seed)
    page_table = np.zeros((B, max_pages), np.int32)
    o = 0
    for b in range(B):
        page_table[b, :npages[b]] = perm[o:o + npages[b]]
        o += npages[b]
    kp = synth.normal((num_pages, Hkv, PAGE, D), seed + 1, device="cuda")
    vp = synth.normal((num_pages, Hkv, PAGE, D), seed + 2, device="cuda")
    cu_q = synth.cu_seqlens(q_lens)
    q = synth.normal((int(cu_q[-1]), Hq, D), seed + 3, device="cuda")
    sink = synth.sink_logits(Hq, seed + 4, device="cuda")
    return ctx, page_table, kp, vp, cu_q, q, sink


def _history_of(b, L, page_table, pool):
    idx = torch.from_numpy(page_table[b, :(L + PAGE - 1) // PAGE].astype(np.int64)).cuda()
    h = pool[idx].transpose(1, 2).reshape(-1, Hkv, D)[:L]   # [L,Hkv,D] by position
    return h.cpu()


@pytest.mark.parametrize("name", ["cfg4_64req", "cfg5_long"])
def test_full_size_verify_sampled(name):
    if name == "cfg4_64req":
        ctx = synth.context_lengths(64, 4096, 65536, 1004)
        q_lens = np.full(64, 4, np.int32)
        sample = [0, 17, 63]
    else:
        ctx = np.full(8, 262144, np.int32)
        q_lens = np.array([4, 1, 4, 1, 4, 1, 4, 1], np.int32)
        sample = [0, 1]
    ctx, page_table, kp, vp, cu_q, q, sink = _full_problem(ctx, q_lens, 1005)
    max_ctx = int(ctx.max())
    o = A.attn_ga_sink_verify(q, torch.from_numpy(cu_q).cuda(), kp, vp,
                              torch.from_numpy(page_table).cuda(), torch.from_numpy(ctx).cuda(),
                              sink, max_ctx=max_ctx, q_max=QMAX)
    assert A.attn_check_device_error() == 0
    assert torch.isfinite(o.float()).all()
    for b in sample:
        L = int(ctx[b])
        kh = _history_of(b, L, page_table, kp)[None]
        vh = _history_of(b, L, page_table, vp)[None]
        r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
        r = oracle.verify(q[r0:r1].cpu(), np.array([0, r1 - r0], np.int32), kh, vh,
                          np.array([L], np.int32), sink.cpu(), None)
        assert_bf16_close(o[r0:r1], r, f"{name} request {b}")


def test_full_size_ring_verify_all_requests():
    """The ring verify at the measured configuration: 64 requests x 4 tokens,
    contexts ~ U[4096, 65536], 131-slot rings filled on the device.  The
    queries see only the last 131 positions, so each request's history for
    the oracle is its ring read out in position order (positions L-131..L-1,
    re-based to 0..130, which keeps every query-key distance)."""
    nreq = 64
    ctx = synth.context_lengths(nreq, 4096, 65536, 2099)
    q_lens = np.full(nreq, QMAX, np.int32)
    cu_q = synth.cu_seqlens(q_lens)
    rk = synth.normal((nreq, Hkv, R, D), 2004, device="cuda")
    rv = synth.normal((nreq, Hkv, R, D), 2005, device="cuda")
    q = synth.normal((nreq * QMAX, Hq, D), 2104, device="cuda")
    sink = synth.sink_logits(Hq, 2105, device="cuda")
    o = A.attn_swa_sink_verify(q, torch.from_numpy(cu_q).cuda(), rk, rv,
                               torch.from_numpy(ctx).cuda(), sink, window=W, q_max=QMAX)
    assert A.attn_check_device_error() == 0
    order = np.stack([(int(L) - R + np.arange(R)) % R for L in ctx])   # slot of position L-R+j
    idx = torch.from_numpy(order).long().cuda()
    kh = torch.stack([rk[b][:, idx[b]] for b in range(nreq)]).transpose(1, 2).cpu()
    vh = torch.stack([rv[b][:, idx[b]] for b in range(nreq)]).transpose(1, 2).cpu()
    ref_o = oracle.verify(q.cpu(), cu_q, kh, vh, np.full(nreq, R, np.int32), sink.cpu(), W)
    assert_bf16_close(o, ref_o, "ring verify, 64 requests x q4")
