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


# ---- the count exchange of a path spread over P processes (one rank each) ----

def _exchange_worker(rank, world, port, q, P, E, T, K, A):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np

        import oracle
        from combine_moe_layout_02_gb300 import inputs, moe

        w = inputs.make(P, E, T, 64, K, seed=9, mask_frac=0.1, expert_alignment=A)
        # This process is source rank `rank` and sees only its own tokens. Its
        # layout row is row 0 of the layout of a routing whose first T tokens
        # are its tokens and whose other tokens are all masked (the oracle
        # stands in for moe_layout on this rank's GPU).
        mine = w.topk_idx[rank * T:(rank + 1) * T]
        lay = oracle.layout(P, E, np.concatenate([mine] + [np.full_like(mine, -1)] * (P - 1)))
        shape = moe.make_shape(P, E, P * T, K, 64, expert_alignment=A)
        plan = moe.exchange_counts(shape, lay["num_tokens_per_rank"][0], lay["num_tokens_per_expert"][0])
        q.put((rank, {k: v.tolist() for k, v in plan.items()}))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("A", [1, 4])
def test_two_rank_count_exchange_matches_notify(A):
    """Two gloo processes, each one expert-parallel rank with its own tokens:
    the all-gathered counts and the plan each computes equal the oracle's
    notify over the whole routing (rank prefix, receive counts, this rank's
    expert counts and offsets, the packed bases), and each rank's send bases
    are the previous rank's prefix row."""
    import numpy as np

    import oracle
    from combine_moe_layout_02_gb300 import inputs

    P, E, T, K = 2, 16, 200, 4
    world = P
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_exchange_worker, args=(r, world, port, q, P, E, T, K, A)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    plans = dict(q.get(timeout=5) for _ in range(world))
    w = inputs.make(P, E, T, 64, K, seed=9, mask_frac=0.1, expert_alignment=A)
    lay = oracle.layout(P, E, w.topk_idx)
    nt = oracle.notify(P, E, w.C, A, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    for r in range(P):
        pl = {k: np.array(v) for k, v in plans[r].items()}
        np.testing.assert_array_equal(pl["ntpr_all"], lay["num_tokens_per_rank"])
        np.testing.assert_array_equal(pl["ntpe_all"], lay["num_tokens_per_expert"])
        np.testing.assert_array_equal(pl["rank_prefix_matrix"], nt["rank_prefix_matrix"])
        np.testing.assert_array_equal(pl["num_recv_tokens"], nt["num_recv_tokens"])
        np.testing.assert_array_equal(pl["num_recv_tokens_per_expert"], nt["num_recv_tokens_per_expert"][r])
        np.testing.assert_array_equal(pl["recv_expert_offset"], nt["recv_expert_offset"][r])
        np.testing.assert_array_equal(pl["part_row_base"], nt["part_row_base"])
        prev = nt["rank_prefix_matrix"][r - 1] if r > 0 else np.zeros(P, np.int64)
        np.testing.assert_array_equal(pl["send_row_base"], prev)
        # send_head rows of rank r's tokens start at its send bases: the
        # smallest send_head entry of its tokens bound for d is the base.
        sh = nt["send_head"][r * T:(r + 1) * T]
        for d in range(P):
            col = sh[:, d][sh[:, d] >= 0]
            if col.size:
                assert col.min() == pl["send_row_base"][d]


def test_exchange_plan_single_process_larger_shapes():
    """The host plan against the oracle's notify for every rank of a P = 8 and
    a P = 128 routing (Zipf, masked), no process group involved."""
    import numpy as np

    import oracle
    from combine_moe_layout_02_gb300 import inputs, moe

    for name, T in (("p8_e256_t4096_h7168", 64), ("p128_e256_t512_h7168_zipf", 8)):
        w = inputs.workload(name, T=T, with_x=False)
        lay = oracle.layout(w.P, w.E, w.topk_idx)
        nt = oracle.notify(w.P, w.E, w.C, w.expert_alignment, lay["num_tokens_per_rank"],
                           lay["num_tokens_per_expert"], lay["is_token_in_rank"])
        shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment)
        for r in (0, 1, w.P - 1):
            pl = moe.moe_exchange_plan(shape, r, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"])
            np.testing.assert_array_equal(pl["rank_prefix_matrix"], nt["rank_prefix_matrix"])
            np.testing.assert_array_equal(pl["part_row_base"], nt["part_row_base"])
            np.testing.assert_array_equal(pl["num_recv_tokens_per_expert"], nt["num_recv_tokens_per_expert"][r])
            np.testing.assert_array_equal(pl["recv_expert_offset"], nt["recv_expert_offset"][r])
    bad = moe.make_shape(2, 4, 4, 1, 8)
    with pytest.raises(moe.MoeError):
        moe.moe_exchange_plan(bad, 2, np.zeros((2, 2)), np.zeros((2, 4)))
    with pytest.raises(moe.MoeError):
        moe.moe_exchange_plan(bad, 0, -np.ones((2, 2)), np.zeros((2, 4)))
