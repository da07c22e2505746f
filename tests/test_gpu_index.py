"""Bit-exact index dumps: the kernels' own tile schedules, masks, ring-slot and
page mappings (the same device functions the kernels run) against the integer
definitions in oracle.index."""
import numpy as np
import pytest
import torch

import synth
from oracle import index

A = pytest.importorskip("global_attention_sinks_swa_b300")
pytestmark = pytest.mark.gpu


def _expected_visits(T, window):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    vis = j <= i
    if window and window > 0:
        vis &= j >= i - window + 1
    return vis.astype(np.int32)


@pytest.mark.parametrize("T,window", [(1, 0), (300, 0), (513, 0), (700, 128), (400, 1),
                                      (389, 200), (256, 129)])
def test_ga_tiling_visits_each_visible_pair_once(T, window):
    got = A.attn_debug_prefill_visits(T, window, mode=0).cpu().numpy()
    np.testing.assert_array_equal(got, _expected_visits(T, window))


@pytest.mark.parametrize("T,window,G", [(16, 128, 8), (500, 128, 8), (333, 120, 8), (300, 64, 4),
                                        (129, 128, 1), (77, 3, 2)])
def test_packed_swa_tiling_visits_each_visible_pair_once(T, window, G):
    got = A.attn_debug_prefill_visits(T, window, mode=1, G=G).cpu().numpy()
    np.testing.assert_array_equal(got, _expected_visits(T, window))


@pytest.mark.parametrize("B,T,Hkv,window,grid", [
    (1, 16, 1, 128, 0),      # one tile
    (1, 500, 1, 128, 3),     # runs of ~10 tiles: the 12-block ring wraps
    (2, 333, 2, 120, 5),     # runs cross (b, kv head) boundaries, ragged tail
    (1, 1000, 2, 114, 7),    # narrowest window of the kernel
    (2, 700, 3, 129, 0),     # widest window, the kernel's own grid
    (1, 2048, 1, 128, 1),    # one CTA streams all 128 tiles
])
def test_swa_stream_schedule_visits_each_visible_pair_once(B, T, Hkv, window, grid):
    """The streaming SWA kernel's run partition, ring-slot bookkeeping and
    column masks, replayed: every visible (query, key) pair exactly once, no
    other pair, no key outside the sequence."""
    got = A.attn_debug_swa_stream_visits(B, T, Hkv, window, grid).cpu().numpy()
    exp = _expected_visits(T, window)
    for bg in range(B * Hkv):
        np.testing.assert_array_equal(got[bg, :, :T], exp, err_msg=f"bg={bg}")
        assert not got[bg, :, T].any(), f"bg={bg}: admitted keys outside [0, T)"


@pytest.mark.parametrize("window,q_max", [(128, 4), (8, 4), (5, 1)])
def test_ring_positions_bit_exact(window, q_max):
    R = index.ring_slots(window, q_max)
    seq_lens = np.array([1, 2, 5, R - 1, R, R + 1, 1000, 1001, 1002, 1003], np.int32)
    q_lens = np.minimum(seq_lens, np.array([1, 2, 4, 4, 3, 4, 4, 1, 2, 3]) % (q_max + 1) + 0)
    q_lens = np.maximum(np.minimum(q_lens, q_max), 1).astype(np.int32)
    cu_q = synth.cu_seqlens(q_lens)
    got = A.attn_debug_verify_positions(0, torch.from_numpy(cu_q).cuda(),
                                        torch.from_numpy(seq_lens).cuda(), q_max, window,
                                        ring_slots=R).cpu().numpy()
    for b, (L, ql) in enumerate(zip(seq_lens, q_lens)):
        for t in range(q_max):
            exp = np.full(R, -1, np.int32)
            if t < ql:
                i = L - ql + t
                for p in range(0, i + 1):
                    if index.visible(i, p, window):
                        exp[index.ring_slot(p, R)] = p
            np.testing.assert_array_equal(got[b, t], exp, err_msg=f"b={b} t={t}")


def test_paged_positions_bit_exact():
    PAGE, q_max = 64, 4
    seq_lens = np.array([1, 64, 65, 4096, 4097, 9000], np.int32)
    q_lens = np.array([1, 4, 2, 4, 3, 4], np.int32)
    max_pages = int((seq_lens.max() + PAGE - 1) // PAGE)
    cu_q = synth.cu_seqlens(q_lens)
    got = A.attn_debug_verify_positions(1, torch.from_numpy(cu_q).cuda(),
                                        torch.from_numpy(seq_lens).cuda(), q_max, 0,
                                        max_pages=max_pages, page_size=PAGE).cpu().numpy()
    n = max_pages * PAGE
    for b, (L, ql) in enumerate(zip(seq_lens, q_lens)):
        for t in range(q_max):
            exp = np.full(n, -1, np.int32)
            if t < ql:
                i = L - ql + t
                exp[:i + 1] = np.arange(i + 1)
            np.testing.assert_array_equal(got[b, t], exp, err_msg=f"b={b} t={t}")
