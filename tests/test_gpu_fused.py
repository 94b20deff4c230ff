"""moe_dispatch_fused (layout + notify + dispatch in one cooperative launch)
against the oracle: every table and every written slot bit-exact, and the
usual combine on its outputs."""

import numpy as np
import pytest

from combine_moe_layout_02_gb300 import inputs, moe
from tests import gpu_path as gp

pytestmark = pytest.mark.gpu


def _run_fused(w, weights=True, repeat=1):
    import torch

    dev = torch.device("cuda", 0)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0)
    buf = moe.Buffers(shape, dev)
    x = torch.from_numpy(w.x_bits.view(np.int16)).to(dev)
    idx = torch.from_numpy(w.topk_idx).to(dev)
    wts = torch.from_numpy(w.topk_weights).to(dev)
    out = torch.empty((w.S, w.H), dtype=torch.int16, device=dev)
    res = {}
    for _ in range(repeat):
        buf.recv_arena.zero_()
        buf.recv_src_idx.fill_(-7)
        buf.recv_topk_idx.fill_(-7)
        buf.recv_topk_weights.fill_(-7.0)
        buf.err.fill_(99)
        buf.dispatch_fused(x, idx, wts)
        torch.cuda.synchronize()
        res["err"] = int(buf.err[0].item())
        buf.combine(out, idx, wts if weights else None)
        torch.cuda.synchronize()
        snap = {k: getattr(buf, k).cpu().numpy() for k in gp.LAYOUT_KEYS + gp.NOTIFY_KEYS}
        snap["is_token_in_rank_bits"] = snap["is_token_in_rank_bits"].view(np.uint32)
        snap["out"] = out.cpu().numpy().view(np.uint16)
        res.setdefault("runs", []).append(snap)
        res.update(snap)
    res.update(buf=buf, y=buf.recv_arena, y_stride=buf.stride, y_rows=buf.arena_rows)
    return res


def _check_fused(w, weights=True, sample=None):
    gpu = _run_fused(w, weights=weights)
    assert gpu["err"] == 0
    lay, nt = gp.oracle_tables(w)
    gp.assert_tables_equal(gpu, lay, nt)
    tokens = None
    if sample is not None and sample < w.S:
        tokens = np.unique(np.concatenate([[0, w.S - 1], np.random.default_rng(1).choice(w.S, sample, False)]))
    gp.compare_dispatch(w, 0, gpu, nt, tokens=tokens)
    gp.compare_combine(w, gpu, nt, tokens=tokens, weights=weights)
    return gpu


def test_fused_tiny():
    _check_fused(inputs.workload("tiny_p4_e16_h256"))


@pytest.mark.parametrize("name,T", [("p32_e256_t128_h1024", None), ("p32_e256_t128_h7168", None),
                                    ("p32_e256_t128_h4096", None), ("p8_e256_t4096_h7168", 300),
                                    ("p8_e256_t4096_h7168", None), ("p32_e256_t128_h2048", 37)])
def test_fused_workloads(name, T):
    _check_fused(inputs.workload(name, T=T), sample=600 if T is None else None)


@pytest.mark.parametrize("P,E,T,K,H,C,A", [
    (1, 8, 333, 4, 64, 16, 1),
    (3, 12, 50, 4, 136, 5, 3),
    (64, 1024, 6, 16, 8192, 16, 2),
    (5, 5, 77, 5, 8, 200, 1),
])
def test_fused_edge_shapes(P, E, T, K, H, C, A):
    _check_fused(inputs.make(P, E, T, H, K, seed=P * 7 + K, mask_frac=0.05, C=C, expert_alignment=A))


def test_fused_out_of_range_ids_and_unit_weights():
    w = inputs.make(4, 16, 64, 64, 2, seed=8)
    w.topk_idx[3, 0] = 16
    gpu = _run_fused(w)
    assert gpu["err"] == moe.MOE_ERR_TOPK_OUT_OF_RANGE
    masked = w.topk_idx.copy()
    masked[masked >= 16] = -1
    lay, nt = gp.oracle_tables(w, topk_idx=masked)
    gp.assert_tables_equal(gpu, lay, nt)
    w2 = inputs.make(8, 64, 40, 256, 6, seed=5, mask_frac=0.2)
    _check_fused(w2, weights=False)


def test_fused_repeat_is_deterministic_and_matches_separate_calls():
    w = inputs.workload("p32_e256_t128_h1024")
    gpu = _run_fused(w, repeat=2)
    a, b = gpu["runs"]
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    sep = gp.run_gpu(w)
    for k in gp.LAYOUT_KEYS + gp.NOTIFY_KEYS + ("out",):
        np.testing.assert_array_equal(a[k], sep[k], err_msg=k)


def test_fused_refuses_large_shapes():
    import torch

    shape = moe.make_shape(128, 256, 128 * 4, 8, 256)
    buf = moe.Buffers(shape, "cuda")
    x = torch.zeros((shape.S, shape.H), dtype=torch.int16, device="cuda")
    idx = torch.zeros((shape.S, shape.K), dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        buf.dispatch_fused(x, idx, None)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


def test_fused_no_tokens():
    """S = 0: every table is still written (zeros), nothing is copied, err 0."""
    import torch

    shape = moe.make_shape(4, 16, 0, 2, 64, 16, 1, 0)
    buf = moe.Buffers(shape, "cuda")
    x = torch.empty((0, 64), dtype=torch.int16, device="cuda")
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    wts = torch.empty((0, 2), dtype=torch.float32, device="cuda")
    for t in (buf.num_tokens_per_rank, buf.num_tokens_per_expert, buf.rank_prefix_matrix,
              buf.num_recv_tokens, buf.num_recv_tokens_per_expert, buf.recv_expert_offset):
        t.fill_(-5)
    buf.part_row_base.fill_(-5)
    buf.err.fill_(99)
    buf.dispatch_fused(x, idx, wts)
    torch.cuda.synchronize()
    assert int(buf.err[0].item()) == 0
    for t in (buf.num_tokens_per_rank, buf.num_tokens_per_expert, buf.rank_prefix_matrix,
              buf.num_recv_tokens, buf.num_recv_tokens_per_expert, buf.recv_expert_offset, buf.part_row_base):
        assert (t.cpu().numpy() == 0).all()


def test_fused_grid_barrier_times_out_and_the_context_stays_usable():
    """The fused launch's bounded grid barrier, made to run out: with the test
    hook one CTA leaves out its arrival and the barrier gives up after 10^4
    polls. Every CTA records MOE_ERR_DEVICE_TIMEOUT, drains its own row loads
    and returns (no trap, no fault, nothing left waiting); a normal fused call
    on the same stream right after is bit-exact with the oracle."""
    import time

    import torch

    w = inputs.workload("p32_e256_t128_h1024", T=32)
    dev = torch.device("cuda", 0)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0)
    buf = moe.Buffers(shape, dev)
    x = torch.from_numpy(w.x_bits.view(np.int16)).to(dev)
    idx = torch.from_numpy(w.topk_idx).to(dev)
    wts = torch.from_numpy(w.topk_weights).to(dev)
    for skip in (0, 5):
        buf.err.fill_(0)
        moe.moe_test_fused_barrier(10_000, skip)
        t0 = time.perf_counter()
        buf.dispatch_fused(x, idx, wts)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 10.0
        assert int(buf.err[0].item()) == moe.MOE_ERR_DEVICE_TIMEOUT
    # the hook armed one call only: this one runs normally
    gpu = _check_fused(w)
    assert gpu["err"] == 0


def test_fused_test_hook_rejects_a_zero_limit():
    with pytest.raises(moe.MoeError):
        moe.moe_test_fused_barrier(0, 0)
