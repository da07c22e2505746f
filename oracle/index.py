"""Integer definitions behind the masks and the cache layouts.

TEST INFRASTRUCTURE ONLY.  The CUDA kernels must reproduce these bit for bit
(checked by the index-dump tests).

- visibility: key position j is visible from query position i iff
  0 <= j <= i and, for a sliding-window layer, j >= i - W + 1 (W keys
  including the query itself).  Window W = 128: MiMo-V2-Flash
  technical-report summary, section "MiMo-V2-Flash Model Architecture".
- SWA ring buffer: a sliding-window layer keeps a fixed-size cache
  (release announcement, section "将效率推向极限").  For MTP verify with up to
  q_max new tokens the ring holds R = W + q_max - 1 slots (131 for W = 128,
  q_max = 4), the union of the windows of the q_max queries; position p lives
  in slot p mod R.  With L positions written, the ring holds positions
  max(0, L - R) .. L - 1.
- GA paged cache: position p of request b lives in page
  page_table[b, p // P] at offset p % P (P = 64 tokens per page).
"""
from __future__ import annotations

import numpy as np


def visible(i: int, j: int, window: int | None) -> bool:
    if j < 0 or j > i:
        return False
    return window is None or window <= 0 or j >= i - window + 1


def ring_slots(window: int, q_max: int) -> int:
    return window + q_max - 1


def ring_slot(p: int, R: int) -> int:
    return p % R


def ring_position_of_slot(slot: int, L: int, R: int) -> int:
    """The position held in `slot` after positions 0..L-1 were written, or -1."""
    for p in range(max(0, L - R), L):
        if p % R == slot:
            return p
    return -1


def page_location(page_table: np.ndarray, b: int, p: int, page_size: int) -> tuple[int, int]:
    return int(page_table[b, p // page_size]), p % page_size


def verify_query_positions(seq_len: int, q_len: int) -> np.ndarray:
    """Positions of the q_len new query tokens of a request of length seq_len."""
    return np.arange(seq_len - q_len, seq_len)
