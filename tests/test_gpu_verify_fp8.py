"""8-bit (E4M3) GA paged cache: the append kernel's codes bit for bit against
oracle.fp8.quantize, and the verify kernel (through the C ABI) against
oracle.verify_fp8 (the plain definition over the dequantized history), on
small mixed problems, split-KV contexts, extreme sinks and the full 64-request
workload on sampled requests."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_bf16_close
from test_gpu_verify import PAGE, QMAX, Hkv, Hq, D, pages_from_history, _history_of

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu


def make_problem(seq_lens, q_lens, seed, extra_pages=3):
    seq_lens = np.asarray(seq_lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    B, Lmax = len(seq_lens), int(seq_lens.max())
    kc = synth.e4m3_codes((B, Lmax, Hkv, D), seed)
    vc = synth.e4m3_codes((B, Lmax, Hkv, D), seed + 1)
    cu_q = synth.cu_seqlens(q_lens)
    q = synth.normal((int(cu_q[-1]), Hq, D), seed + 2)
    sink = synth.sink_logits(Hq, seed + 3)
    ks, vs = synth.kv_scales(Hkv, seed + 5), synth.kv_scales(Hkv, seed + 6)
    max_pages = (Lmax + PAGE - 1) // PAGE
    num_pages = B * max_pages + extra_pages
    perm = synth.page_permutation(num_pages, seed + 4)
    page_table = perm[:B * max_pages].reshape(B, max_pages).copy()
    return dict(seq_lens=seq_lens, cu_q=cu_q, q=q, sink=sink, kc=kc, vc=vc, ks=ks, vs=vs,
                page_table=page_table, num_pages=num_pages)


def run(P, sink=None, max_ctx=None):
    sink = P["sink"] if sink is None else sink
    kp = pages_from_history(P["kc"], P["seq_lens"], P["page_table"], P["num_pages"]).cuda()
    vp = pages_from_history(P["vc"], P["seq_lens"], P["page_table"], P["num_pages"]).cuda()
    max_ctx = int(P["seq_lens"].max()) if max_ctx is None else max_ctx
    o = A.attn_ga_sink_verify_fp8(P["q"].cuda(), torch.from_numpy(P["cu_q"]).cuda(), kp, vp,
                                  torch.from_numpy(P["page_table"]).cuda(),
                                  torch.from_numpy(P["seq_lens"]).cuda(), sink.cuda(),
                                  P["ks"].cuda(), P["vs"].cuda(), max_ctx=max_ctx, q_max=QMAX)
    assert A.attn_check_device_error() == 0
    return o


def ref(P, sink=None):
    sink = P["sink"] if sink is None else sink
    return oracle.verify_fp8(P["q"], P["cu_q"], P["kc"].numpy(), P["vc"].numpy(), P["ks"],
                             P["vs"], P["seq_lens"], sink, None)


CASES = [
    ([4, 50, 131, 132, 700], [4, 1, 3, 4, 2]),
    ([1, 2, 3, 4], [1, 2, 3, 4]),
    ([64, 65, 128, 4096, 4097, 9000], [4, 4, 1, 2, 3, 4]),
]


@pytest.mark.parametrize("seq_lens,q_lens", CASES)
def test_fp8_paged_verify(seq_lens, q_lens):
    P = make_problem(seq_lens, q_lens, seed=7 + sum(seq_lens))
    assert_bf16_close(run(P), ref(P), f"fp8 verify {seq_lens}")


def test_fp8_verify_split_paths_agree_and_extreme_sinks():
    P = make_problem([300, 5000, 12000], [4, 2, 3], seed=77)
    sink = P["sink"].clone()
    sink[0], sink[9], sink[10] = math.inf, -math.inf, 30.0
    o1 = run(P, sink)
    o2 = run(P, sink, max_ctx=20000)   # more splits, same result
    r = ref(P, sink)
    assert_bf16_close(o1, r, "fp8 extreme sinks")
    assert_bf16_close(o2, r, "fp8 more splits")


def test_fp8_append_codes_bit_exact():
    """Codes of value / scale[kv head] (fp32 division, round to nearest even,
    saturation beyond 448), written at page_table[b][p/64], offset p%64."""
    B = 3
    seq_lens = np.array([5, 64, 130], np.int32)
    q_lens = np.array([4, 1, 3], np.int32)
    cu_q = synth.cu_seqlens(q_lens)
    rows = int(cu_q[-1])
    k_new = synth.normal((rows, Hkv, D), 901)
    v_new = synth.normal((rows, Hkv, D), 902) * 4
    k_new[0, 0, :8] = torch.tensor([1e4, -1e4, 5.0, -0.0, 0.0, 1e-6, -1e-6, 7.0]).bfloat16()
    ks, vs = synth.kv_scales(Hkv, 903), synth.kv_scales(Hkv, 904)
    max_pages = 3
    num_pages = B * max_pages + 2
    page_table = synth.page_permutation(num_pages, 905)[:B * max_pages].reshape(B, max_pages).copy()
    kp = torch.full((num_pages, Hkv, PAGE, D), 0x55, dtype=torch.uint8, device="cuda")
    vp = kp.clone()
    A.attn_ga_paged_append_fp8(k_new.cuda(), v_new.cuda(), torch.from_numpy(cu_q).cuda(),
                               torch.from_numpy(seq_lens).cuda(), kp, vp,
                               torch.from_numpy(page_table).cuda(), ks.cuda(), vs.cuda(),
                               q_max=QMAX)
    assert A.attn_check_device_error() == 0
    kp, vp = kp.cpu().numpy(), vp.cpu().numpy()
    written = np.zeros(kp.shape[:3], bool)
    for b in range(B):
        for t in range(int(q_lens[b])):
            row, pos = int(cu_q[b]) + t, int(seq_lens[b]) - int(q_lens[b]) + t
            page, off = page_table[b, pos // PAGE], pos % PAGE
            written[page, :, off] = True
            for g in range(Hkv):
                np.testing.assert_array_equal(
                    kp[page, g, off], oracle.fp8.quantize(k_new[row, g].float().numpy(), ks[g].item()))
                np.testing.assert_array_equal(
                    vp[page, g, off], oracle.fp8.quantize(v_new[row, g].float().numpy(), vs[g].item()))
    assert (kp[~written] == 0x55).all() and (vp[~written] == 0x55).all()


def test_full_size_fp8_verify_sampled():
    """64 requests x q4, contexts ~ U[4096, 65536], 8-bit pages filled on the device."""
    ctx = synth.context_lengths(64, 4096, 65536, 1004)
    q_lens = np.full(64, 4, np.int32)
    npages = (ctx + PAGE - 1) // PAGE
    max_pages, num_pages = int(npages.max()), int(npages.sum())
    perm = synth.page_permutation(num_pages, 1105)
    page_table = np.zeros((64, max_pages), np.int32)
    o_ = 0
    for b in range(64):
        page_table[b, :npages[b]] = perm[o_:o_ + npages[b]]
        o_ += npages[b]
    kp = synth.e4m3_codes((num_pages, Hkv, PAGE, D), 1106, device="cuda")
    vp = synth.e4m3_codes((num_pages, Hkv, PAGE, D), 1107, device="cuda")
    cu_q = synth.cu_seqlens(q_lens)
    q = synth.normal((int(cu_q[-1]), Hq, D), 1108, device="cuda")
    sink = synth.sink_logits(Hq, 1109, device="cuda")
    ks, vs = synth.kv_scales(Hkv, 1110, device="cuda"), synth.kv_scales(Hkv, 1111, device="cuda")
    o = A.attn_ga_sink_verify_fp8(q, torch.from_numpy(cu_q).cuda(), kp, vp,
                                  torch.from_numpy(page_table).cuda(), torch.from_numpy(ctx).cuda(),
                                  sink, ks, vs, max_ctx=int(ctx.max()), q_max=QMAX)
    assert A.attn_check_device_error() == 0
    for b in (0, 17, 63):
        L = int(ctx[b])
        kh = _history_of(b, L, page_table, kp)[None].numpy()
        vh = _history_of(b, L, page_table, vp)[None].numpy()
        r0, r1 = int(cu_q[b]), int(cu_q[b + 1])
        r = oracle.verify_fp8(q[r0:r1].cpu(), np.array([0, r1 - r0], np.int32), kh, vh, ks.cpu(),
                              vs.cpu(), np.array([L], np.int32), sink.cpu(), None)
        assert_bf16_close(o[r0:r1], r, f"fp8 full size request {b}")


def test_fp8_bad_page_ids_are_reported():
    """A page id outside the pool sets ATTN_DEVERR_PAGE_OOB in the 8-bit append
    and verify, and the context stays usable."""
    A.attn_check_device_error()
    num_pages = 4
    pt = torch.tensor([[0, 1], [2, 77]], dtype=torch.int32, device="cuda")
    seq_lens = torch.tensor([100, 100], dtype=torch.int32, device="cuda")
    cu_q = torch.tensor([0, 4, 8], dtype=torch.int32, device="cuda")
    kp = torch.zeros(num_pages, Hkv, PAGE, D, dtype=torch.uint8, device="cuda")
    vp = kp.clone()
    ks = torch.full((Hkv,), 0.02, device="cuda")
    new = synth.normal((8, Hkv, D), 1, device="cuda")
    A.attn_ga_paged_append_fp8(new, new.clone(), cu_q, seq_lens, kp, vp, pt, ks, ks, q_max=QMAX)
    assert A.attn_check_device_error() & A.DEVERR_PAGE_OOB
    q = synth.normal((8, Hq, D), 2, device="cuda")
    sink = synth.sink_logits(Hq, 3, device="cuda")
    A.attn_ga_sink_verify_fp8(q, cu_q, kp, vp, pt, seq_lens, sink, ks, ks, max_ctx=128, q_max=QMAX)
    assert A.attn_check_device_error() & A.DEVERR_PAGE_OOB
    assert A.attn_check_device_error() == 0
    assert torch.isfinite(torch.ones(4, device="cuda").sum())
