"""Host logic of the multi-process benchmark on CPU (gloo, world size 2):
ranks read their identity from the environment, time independently, and the
reported time is the maximum over ranks; value counts the units of all ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_env()
    bench.barrier(w)
    t = bench.reduce_max(1.0 + rank * 0.5, w)          # per-rank "ms per step"
    flop = bench.prefill_flop(bench.T, bench.W)
    value = w * flop / (t * 1e-3) / 1e12
    q.put((r, w, local, t, value))
    dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == pytest.approx(1.5) for r in res)          # max over ranks
    single = 1 * __import__("bench").prefill_flop(32768, 128) / 1.5e-3 / 1e12
    assert res[0][4] == pytest.approx(2 * single)                  # both ranks' units


def test_workload_counts():
    import bench
    assert bench.visible_pairs(32768, 128) == 128 * 32768 - 8128
    assert bench.visible_pairs(32768, None) == 32768 * 32769 // 2
    assert bench.prefill_flop(32768, 128) == pytest.approx(1.3717e11, rel=1e-4)
    assert bench.prefill_flop(32768, None) == pytest.approx(1.7593e13, rel=1e-4)
    assert bench.prefill_min_bytes() == pytest.approx(1.208e9, rel=1e-3)
