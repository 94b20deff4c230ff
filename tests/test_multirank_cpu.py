"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks run
independent replicas; the reported time is the maximum over ranks and the
units are summed."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        assert bench.dist_env() == (world, rank, rank)
        bench.barrier(world)
        t, u = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), world)
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_max_time_sum_units():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, t, u in res:
        assert t == pytest.approx(2.0)
        assert u == pytest.approx(300.0)


def test_single_rank_is_identity():
    import bench

    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_algorithmic_bytes_formulas():
    import bench

    # One token, one rank, H = 8, K = 1: read 16 B, write 16 + 12 + 4 + 8, ids 8, send_head 4.
    assert bench.dispatch_bytes(1, 1, 1, 8, 1, 0) == 16 + (16 + 12) + 4 + 8 + 8 + 4
    assert bench.combine_bytes(1, 1, 1, 8, 1) == 16 + 16 + 4 + 8


@pytest.mark.parametrize("layout", ["rank", "expert"])
def test_cpu_baseline_runs_on_int8_workloads(layout):
    """The oracle leg of the int8 workload: combine reads a bf16 stand-in
    arena (the int8 slots are not bf16 rows)."""
    import bench

    tps, passes, secs, sample = bench.oracle_sample("p8_e256_t4096_h7168_int8", 8, 0.0, max_passes=1,
                                                    layout=layout)
    assert passes == 1 and tps > 0 and "T=8" in sample
    assert bench.oracle_sample.last["quant"] == 1


def test_oracle_combine_refuses_a_short_arena():
    import numpy as np

    import oracle

    P, E, H, S, K = 2, 4, 8, 2, 1
    y = np.zeros((3, 2 * H), np.uint8)  # 3 rows of 16 bytes
    send_head = np.zeros((S, P), np.int32)
    idx = np.zeros((S, K), np.int32)
    prb = np.array([0, 1, 4], np.int64)
    with pytest.raises(ValueError):
        oracle.combine(P, E, H, y, 2 * H, prb, 4, send_head, idx, None)
    with pytest.raises(ValueError):
        oracle.combine(P, E, H, y, H, prb, 3, send_head, idx, None)
