"""Index logic of the kernels replayed on the CPU, from the kernels' own
functions (index_math.cuh compiled as host code):
- the streaming SWA prefill schedule must admit every visible (query, key)
  pair exactly once across the CTA runs and the shared-memory ring of 16-key
  blocks, and never need more live blocks than the ring holds, for batches of
  equal length and for packed batches (cu_seqlens);
- the ring verify's visible slots (two slot intervals) must be exactly the
  slots holding positions in the query's window;
- the GA prefill's block order must cover every (pair, head, sequence) once,
  with the heads of one kv head adjacent and the heaviest pairs first.
No GPU needed; the same functions run on the device in test_gpu_index."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host", "swa_schedule_replay.cu")
INC = os.path.join(ROOT, "global_attention_sinks_swa_b300", "csrc")
LIB = os.path.join(ROOT, "_build", "libswa_schedule_replay.so")
RING_BLOCKS = 12


@pytest.fixture(scope="module")
def replay():
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    deps = [SRC, os.path.join(INC, "index_math.cuh")]
    if not os.path.exists(LIB) or any(os.path.getmtime(d) > os.path.getmtime(LIB) for d in deps):
        nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
        subprocess.run([nvcc, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", INC,
                        SRC, "-o", LIB], check=True)
    lib = ctypes.CDLL(LIB)
    f = lib.swa_stream_visits_host
    f.argtypes = [np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS"), ctypes.c_void_p] + \
        [ctypes.c_int] * 6
    f.restype = ctypes.c_int
    lib.ring_visible_host.argtypes = [np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")] + [ctypes.c_int] * 4
    lib.ring_visible_host.restype = None

    def run(B, T, Hkv, window, grid, cu=None):
        """cu: packed batch offsets [B+1] (T = the longest sequence), or None."""
        visits = np.zeros((B * Hkv, T, T + 1), np.int32)
        if cu is None:
            live = f(visits, None, B, T, B * T, Hkv, window, grid)
        else:
            cu = np.ascontiguousarray(cu, np.int32)
            live = f(visits, cu.ctypes.data_as(ctypes.c_void_p), B, T, int(cu[-1]), Hkv, window,
                     grid)
        return visits, live
    run.ring_visible = lib.ring_visible_host
    lib.ga_block_coords_host.argtypes = [np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")] + \
        [ctypes.c_int] * 4
    lib.ga_block_coords_host.restype = None
    run.ga_block_coords = lib.ga_block_coords_host
    return run


def _expected(T, window):
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    return ((j <= i) & (j >= i - window + 1)).astype(np.int32)


@pytest.mark.parametrize("B,T,Hkv,window,grid", [
    (1, 1, 1, 128, 1), (1, 16, 1, 128, 1), (1, 17, 1, 128, 2), (1, 500, 1, 128, 3),
    (2, 333, 2, 120, 5), (1, 1000, 2, 114, 7), (2, 700, 3, 129, 148), (1, 2048, 1, 128, 1),
    (3, 257, 2, 128, 4), (1, 3000, 2, 128, 148),
])
def test_schedule_admits_each_visible_pair_once(replay, B, T, Hkv, window, grid):
    nblk = (T + 15) // 16
    grid = min(grid, nblk * Hkv * B)
    visits, live = replay(B, T, Hkv, window, grid)
    exp = _expected(T, window)
    for bg in range(B * Hkv):
        np.testing.assert_array_equal(visits[bg, :, :T], exp, err_msg=f"bg={bg}")
        assert not visits[bg, :, T].any()
    assert live <= RING_BLOCKS


@pytest.mark.parametrize("lens,Hkv,window,grid", [
    ([5, 0, 40, 16, 17], 2, 128, 3), ([300, 1, 0, 0, 129], 1, 128, 148),
    ([0, 0, 7], 3, 120, 2), ([1000, 200, 33], 2, 114, 7), ([2], 1, 129, 1),
])
def test_packed_schedule_admits_each_visible_pair_once(replay, lens, Hkv, window, grid):
    """Packed batches: each sequence starts its own tile grid; keys outside the
    sequence (before its first token or past its end) are never admitted, and
    empty sequences take no tiles."""
    B, T = len(lens), max(max(lens), 1)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ntiles = Hkv * sum((n + 15) // 16 for n in lens)
    visits, live = replay(B, T, Hkv, window, max(1, min(grid, ntiles)), cu)
    for b, n in enumerate(lens):
        exp = _expected(n, window)
        for g in range(Hkv):
            v = visits[b * Hkv + g]
            np.testing.assert_array_equal(v[:n, :n], exp, err_msg=f"b={b} g={g}")
            assert not v[:n, n:].any() and not v[n:].any()
    assert live <= RING_BLOCKS


def test_packed_equal_lengths_match_the_unpacked_replay(replay):
    lens = [123, 123, 123]
    cu = np.array([0, 123, 246, 369], np.int32)
    a, la = replay(3, 123, 2, 128, 5)
    b, lb = replay(3, 123, 2, 128, 5, cu)
    np.testing.assert_array_equal(a, b)
    assert la == lb


def test_replay_catches_a_wrong_window(replay):
    """A schedule built for W=128 does not pass as W=127 (the check has teeth)."""
    visits, _ = replay(1, 300, 1, 128, 2)
    assert not np.array_equal(visits[0, :, :300], _expected(300, 127))


def test_ring_visible_slots_match_the_definition(replay):
    """Slot s of a ring of R slots, after positions 0..L-1 were written, holds
    the p in [L-R, L) with p = s mod R; it is visible from query position i iff
    max(0, i-W+1) <= p <= i."""
    rng = np.random.default_rng(7)
    for _ in range(3000):
        q_max = int(rng.integers(1, 5))
        W = int(rng.integers(1, 142))
        R = W + q_max - 1 + int(rng.integers(0, 3))
        L = int(rng.integers(1, 4 * R + 10))
        q_len = int(rng.integers(1, min(q_max, L) + 1))
        t = int(rng.integers(0, q_len))
        i = L - q_len + t
        got = np.zeros(R, np.int32)
        replay.ring_visible(got, L, R, W, i)
        exp = np.full(R, -1, np.int32)
        for p in range(max(0, L - R), L):
            if max(0, i - W + 1) <= p <= i:
                exp[p % R] = p
        np.testing.assert_array_equal(got, exp, err_msg=f"L={L} R={R} W={W} i={i}")


@pytest.mark.parametrize("B,T,Hq,Hkv", [(1, 32768, 64, 8), (2, 300, 4, 1), (3, 1000, 6, 2),
                                        (1, 256, 8, 8)])
def test_ga_block_order_is_a_permutation(replay, B, T, Hq, Hkv):
    """Every (pair, head, sequence) of the GA prefill grid comes from exactly
    one block; the G heads of one kv head take consecutive blocks of one pair,
    and within one (kv head, sequence) the pairs run from the last to the first."""
    npairs = (T + 255) // 256
    n = npairs * Hq * B
    out = np.zeros(3 * n, np.int32)
    replay.ga_block_coords(out, n, npairs, Hq, Hkv)
    c = out.reshape(n, 3)
    assert c[:, 0].min() >= 0 and c[:, 0].max() < npairs
    assert c[:, 1].min() >= 0 and c[:, 1].max() < Hq
    assert c[:, 2].min() >= 0 and c[:, 2].max() < B
    keys = (c[:, 2].astype(np.int64) * Hq + c[:, 1]) * npairs + c[:, 0]
    assert len(np.unique(keys)) == n
    G = Hq // Hkv
    groups = c.reshape(n // G, G, 3)
    assert (groups[:, :, 0] == groups[:, :1, 0]).all()          # one pair per group of blocks
    assert (groups[:, :, 1] // G == groups[:, :1, 1] // G).all()  # one kv head per group
    assert (groups[:, :, 1] % G == np.arange(G)).all()
    pairs = groups[:, 0, 0].reshape(B * Hkv, npairs)
    assert (pairs == np.arange(npairs - 1, -1, -1)).all()
