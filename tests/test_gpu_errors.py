"""Failure reporting without a GPU fault: bad inputs that only the device can
see set bits in the device error word (the offending work is skipped, no trap,
no hang), a pipeline wait that nothing completes gives up after its time limit,
and host-detectable errors return a status before any launch."""
import numpy as np
import pytest
import torch

import oracle
import synth

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu

Hq, Hkv, D = 64, 8, 128


def _clear():
    A.attn_check_device_error()


def test_page_id_out_of_pool_sets_bit_and_context_survives():
    _clear()
    B, PAGE, num_pages = 2, 64, 8
    page_table = torch.tensor([[0, 1, 2, 3], [4, 5, 99, 7]], dtype=torch.int32, device="cuda")
    seq_lens = torch.tensor([150, 150], dtype=torch.int32, device="cuda")  # appends land in page index 2
    cu_q = torch.tensor([0, 4, 8], dtype=torch.int32, device="cuda")
    kp = synth.normal((num_pages, Hkv, PAGE, D), 1, device="cuda")
    vp = synth.normal((num_pages, Hkv, PAGE, D), 2, device="cuda")
    q = synth.normal((8, Hq, D), 3, device="cuda")
    sink = synth.sink_logits(Hq, 4, device="cuda")
    A.attn_ga_sink_verify(q, cu_q, kp, vp, page_table, seq_lens, sink, max_ctx=256)
    assert A.attn_check_device_error() & A.DEVERR_PAGE_OOB
    k_new = synth.normal((8, Hkv, D), 5, device="cuda")
    A.attn_ga_paged_append(k_new, k_new.clone(), cu_q, seq_lens, kp, vp, page_table, q_max=4)
    assert A.attn_check_device_error() & A.DEVERR_PAGE_OOB
    # the context is still usable and the word was cleared
    assert A.attn_check_device_error() == 0
    assert torch.isfinite(torch.ones(4, device="cuda").sum())


def test_qlen_above_qmax_and_short_context_set_bits():
    _clear()
    B, R = 2, 131
    ring = synth.normal((B, Hkv, R, D), 1, device="cuda")
    cu_q = torch.tensor([0, 4, 9], dtype=torch.int32, device="cuda")   # second request: 5 > q_max
    seq_lens = torch.tensor([3, 100], dtype=torch.int32, device="cuda")  # first: L < q_len
    q = synth.normal((9, Hq, D), 2, device="cuda")
    sink = synth.sink_logits(Hq, 3, device="cuda")
    A.attn_swa_sink_verify(q, cu_q, ring, ring.clone(), seq_lens, sink, window=128, q_max=4)
    bits = A.attn_check_device_error()
    assert bits & A.DEVERR_QLEN and bits & A.DEVERR_CTX_OOB


def test_wait_timeout_sets_bit_then_launches_skip_until_cleared():
    _clear()
    q, k, v, sink = synth.prefill_inputs(1, 256, Hq, Hkv, D, 17)
    q, k, v, sink = q.cuda(), k.cuda(), v.cuda(), sink.cuda()
    # a wait that nothing completes runs out (about 2 s) and sets the bit
    A.attn_debug_wait_timeout()
    o = torch.full_like(q, float("nan"))
    A.attn_swa_sink_prefill(q, k, v, sink, window=128, out=o)
    assert A.attn_check_device_error() & A.DEVERR_WAIT_TIMEOUT
    assert torch.isnan(o.float()).all()  # launched while the bit was set: no work done
    # reading the word cleared it; the same call now computes
    assert A.attn_check_device_error() == 0
    A.attn_swa_sink_prefill(q, k, v, sink, window=128, out=o)
    assert A.attn_check_device_error() == 0
    ref = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), sink.cpu(), 128)
    assert np.abs(o.float().cpu().numpy() - ref).max() < 2e-2


def test_host_side_errors_return_status():
    q = torch.zeros(1, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, 1, 128, dtype=torch.bfloat16, device="cuda")
    sink = torch.zeros(8, device="cuda")
    with pytest.raises(A.AttnError) as e:
        A.attn_swa_sink_prefill(q, k, k, sink, window=0)
    assert e.value.status == A.ATTN_ERR_INVALID_ARG
    q64 = torch.zeros(1, 16, 8, 64, dtype=torch.bfloat16, device="cuda")
    k64 = torch.zeros(1, 16, 1, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(A.AttnError) as e:
        A.attn_ga_sink_prefill(q64, k64, k64, sink)
    assert e.value.status == A.ATTN_ERR_UNSUPPORTED
    ring = torch.zeros(1, 1, 100, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(A.AttnError) as e:   # ring smaller than window + q_max - 1
        A.attn_swa_sink_verify(torch.zeros(4, 8, 128, dtype=torch.bfloat16, device="cuda"),
                               torch.tensor([0, 4], dtype=torch.int32, device="cuda"), ring, ring,
                               torch.tensor([10], dtype=torch.int32, device="cuda"), sink,
                               window=128, q_max=4)
    assert e.value.status == A.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("entry", ["workspace", "noalloc"])
def test_wait_timeout_skips_split_verify_and_its_merge(entry):
    """Contexts longer than one 4096-token split run the split-KV merge kernel.
    A first call fills the split scratch with valid partials; with the timeout
    bit set, a second call must leave its output untouched rather than merge
    whatever the scratch still holds."""
    _clear()
    ctx = np.array([9000, 5000], np.int32)
    npages = (ctx + 63) // 64
    num_pages = int(npages.sum())
    pt = np.zeros((2, int(npages.max())), np.int32)
    pt[0, :npages[0]] = np.arange(npages[0])
    pt[1, :npages[1]] = npages[0] + np.arange(npages[1])
    kp = synth.normal((num_pages, Hkv, 64, D), 31, device="cuda")
    vp = synth.normal((num_pages, Hkv, 64, D), 32, device="cuda")
    cu_q = torch.tensor([0, 4, 7], dtype=torch.int32, device="cuda")
    q = synth.normal((7, Hq, D), 33, device="cuda")
    sink = synth.sink_logits(Hq, 34, device="cuda")
    args = (q, cu_q, kp, vp, torch.from_numpy(pt).cuda(), torch.from_numpy(ctx).cuda(), sink)
    max_ctx = 12000   # three splits
    assert A.attn_ga_sink_verify_workspace(2, Hq, Hkv, D, 4, max_ctx) > 0
    ws = torch.empty(A.attn_ga_sink_verify_workspace(2, Hq, Hkv, D, 4, max_ctx),
                     dtype=torch.uint8, device="cuda")

    def call(out):
        if entry == "workspace":
            A.attn_ga_sink_verify(*args, max_ctx=max_ctx, q_max=4, out=out, workspace=ws)
        else:
            A.attn_ga_sink_verify_noalloc(*args, max_ctx=max_ctx, q_max=4, out=out)

    good = torch.empty_like(q)
    call(good)   # leaves valid partials in the scratch
    assert A.attn_check_device_error() == 0
    assert torch.isfinite(good.float()).all()
    A.attn_debug_wait_timeout()
    o = torch.full_like(q, float("nan"))
    call(o)
    assert A.attn_check_device_error() & A.DEVERR_WAIT_TIMEOUT
    assert torch.isnan(o.float()).all()   # neither the splits nor the merge wrote anything
    o2 = torch.full_like(q, float("nan"))
    call(o2)   # the word was cleared: the same call computes again
    assert A.attn_check_device_error() == 0
    assert torch.equal(o2, good)
