"""Host-side checks of the cache layouts under an MTP accept/reject walk.

The SWA layer keeps a fixed-size ring of R = W + q_max - 1 slots per request
and kv-head; position p lives in slot p mod R.  A verify pass appends q_len
tokens, the caller accepts a prefix and rolls the sequence length back; the
next append overwrites the rejected slots.  These tests replay such walks on
the CPU with the oracle's index definitions and check that the ring always
holds every key that any query of the next pass can see.
"""
import os

import numpy as np
import pytest

import synth
from oracle import index

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mtp_verify_walk.txt")


def _parse_golden():
    rows = {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            key, val = line.split(":", 1)
            rows[key.strip()] = val.split()
    return rows


def _offset(tok: str) -> int:
    return 0 if tok == "i" else int(tok.split("+")[1])


def test_golden_walk_rollback_rule():
    """After a pass over inputs i..i+3 whose predictions are accept, accept,
    reject, discard, the next pass starts at i + 1 + accepted (the figure's
    i+3): new_len = old_len - q_len + 1 + accepted."""
    g = _parse_golden()
    q_len = len(g["inputs"])
    accepted = 0
    for v in g["verdicts"]:
        if v != "accept":
            break
        accepted += 1
    assert accepted == 2
    start = _offset(g["inputs"][0])
    next_start = start + 1 + accepted
    assert _offset(g["next_inputs"][0]) == next_start
    assert [_offset(t) for t in g["next_inputs"]] == list(range(next_start, next_start + q_len))


def _walk(window, q_max, steps, seed, L0):
    """Replay a walk; return the list of (seq_len, q_len) of each verify pass."""
    acc = synth.accept_counts(steps, q_max, seed)
    g = _parse_golden()
    passes, base = [], L0
    for s in range(steps):
        q_len = q_max if s % 5 != 4 else 1 + (s // 5) % q_max
        passes.append((base + q_len, q_len))
        a = int(acc[s])
        if s == 0:
            a = sum(1 for v in g["verdicts"] if v == "accept")   # the figure's pass first
        base = base + 1 + min(a, q_len - 1)
    return passes


@pytest.mark.parametrize("window,q_max", [(128, 4), (8, 4), (5, 2), (1, 1), (3, 3)])
@pytest.mark.parametrize("L0", [0, 1, 130])
def test_ring_holds_every_visible_key(window, q_max, L0):
    R = index.ring_slots(window, q_max)
    ring = {}                      # slot -> position currently stored
    for seq_len, q_len in _walk(window, q_max, 200, seed=window * 7 + q_max, L0=L0):
        if not ring and L0:
            for p in range(max(0, seq_len - q_len - R), seq_len - q_len):
                ring[index.ring_slot(p, R)] = p
        for p in range(seq_len - q_len, seq_len):            # append the new tokens
            ring[index.ring_slot(p, R)] = p
        for i in index.verify_query_positions(seq_len, q_len):
            for j in range(max(0, i - window - 2), i + 1):
                if index.visible(i, j, window):
                    assert ring.get(index.ring_slot(j, R)) == j, (seq_len, q_len, i, j)
        # slot -> position map used by the kernels: wherever the formula names a
        # position that some query of this pass can see, the ring holds it (a
        # slot may hold a stale rejected draft only where nothing can see it).
        qpos = index.verify_query_positions(seq_len, q_len)
        for slot in range(R):
            p = index.ring_position_of_slot(slot, seq_len, R)
            if p >= 0 and any(index.visible(int(i), p, window) for i in qpos):
                assert ring.get(slot) == p


def test_ring_too_small_is_detected():
    """With one slot fewer than W + q_max - 1 some visible key is overwritten."""
    window, q_max = 8, 4
    R = index.ring_slots(window, q_max) - 1
    seq_len, q_len = 40, 4
    ring = {index.ring_slot(p, R): p for p in range(seq_len)}
    i = seq_len - q_len
    missing = [j for j in range(i - window + 1, i + 1) if ring.get(index.ring_slot(j, R)) != j]
    assert missing
