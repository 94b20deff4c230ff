"""moe_run_host: the path over host-resident batches, end to end, against the oracle.

Each batch's expected rows come from the oracle's layout -> notify -> dispatch
and combine ("HCCL Window 模式 (Non-SHMEM) 代码深度剖析", sections 3.6 and 7.8)
with identity experts (combine reads the dispatch arena), or with given expert
outputs y for the int8 payload.
"""

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs, moe

pytestmark = pytest.mark.gpu


def _batches(P, E, T, H, K, n, quant=0, mask_frac=0.0):
    return [inputs.make(P, E, T, H, K, seed=100 + i, quant=quant, mask_frac=mask_frac) for i in range(n)]


def _expected(w, weights=True, y=None, y_stride=None, arena_rows=None):
    lay, nt, dis = oracle.run_all(w.P, w.E, w.C, w.expert_alignment, w.H, w.quant, w.x_bits, w.topk_idx,
                                  w.topk_weights)
    if y is None:
        y, y_stride, rows = dis["arena"], oracle.slot_stride(w.H, 0), int(nt["part_row_base"][-1])
    else:
        rows = arena_rows
    ref = oracle.combine(w.P, w.E, w.H, y, y_stride, nt["part_row_base"], rows, nt["send_head"], w.topk_idx,
                         w.topk_weights if weights else None)
    assert ref["err"] == 0
    return ref["out"]


def _run(ws, weights=True, fused=False, y=None, y_stride=0, alias_out=False):
    import torch

    w0 = ws[0]
    shape = moe.make_shape(w0.P, w0.E, w0.S, w0.K, w0.H, w0.C, w0.expert_alignment, w0.quant)
    n = len(ws)
    xs = [torch.from_numpy(w.x_bits.view(np.int16)).pin_memory() for w in ws]
    ids = [torch.from_numpy(w.topk_idx).pin_memory() for w in ws]
    wts = [torch.from_numpy(w.topk_weights).pin_memory() for w in ws] if weights else None
    if alias_out:
        one = torch.empty((w0.S, w0.H), dtype=torch.int16).pin_memory()
        outs = [one] * n
    else:
        outs = [torch.empty((w0.S, w0.H), dtype=torch.int16).pin_memory() for _ in ws]
    wsb = moe.moe_run_host_workspace_bytes(shape, n)
    assert wsb > 0
    workspace = torch.empty((wsb,), dtype=torch.uint8, device="cuda")
    err = np.full(n, -1, np.int32)
    moe.moe_run_host(shape, xs, ids, wts, outs, workspace, y=y, y_row_stride=y_stride, fused=fused,
                     err_host=err)
    assert (err == 0).all()
    return [o.numpy().view(np.uint16).copy() for o in outs]


@pytest.mark.parametrize("fused", [False, True])
def test_batches_match_the_oracle(fused):
    ws = _batches(4, 16, 96, 256, 4, 3, mask_frac=0.05)
    got = _run(ws, fused=fused)
    for w, g in zip(ws, got):
        np.testing.assert_array_equal(g, _expected(w))


def test_unit_weights_and_ragged_shape():
    ws = _batches(5, 20, 37, 72, 3, 4)
    got = _run(ws, weights=False)
    for w, g in zip(ws, got):
        np.testing.assert_array_equal(g, _expected(w, weights=False))


def test_many_batches_with_aliased_output_keep_the_last():
    ws = _batches(8, 64, 64, 512, 8, 5)
    got = _run(ws, alias_out=True)
    np.testing.assert_array_equal(got[-1], _expected(ws[-1]))


def test_int8_payload_with_expert_outputs():
    import torch

    ws = _batches(4, 16, 64, 256, 4, 3, quant=1)
    w0 = ws[0]
    shape = moe.make_shape(w0.P, w0.E, w0.S, w0.K, w0.H, w0.C, w0.expert_alignment, 1)
    rows = moe.moe_max_recv_rows(shape)
    gen = torch.Generator(device="cuda").manual_seed(7)
    y = torch.empty((rows, w0.H), dtype=torch.bfloat16, device="cuda").normal_(generator=gen).view(torch.int16)
    got = _run(ws, y=y, y_stride=2 * w0.H)
    y_host = y.cpu().numpy().view(np.uint16)
    for w, g in zip(ws, got):
        np.testing.assert_array_equal(g, _expected(w, y=y_host, y_stride=2 * w.H, arena_rows=rows))


def test_device_errors_are_reported_per_batch():
    import torch

    ws = _batches(4, 16, 32, 64, 2, 3)
    ws[1].topk_idx[3, 0] = 16  # expert id >= E in batch 1
    w0 = ws[0]
    shape = moe.make_shape(w0.P, w0.E, w0.S, w0.K, w0.H, w0.C, w0.expert_alignment, 0)
    xs = [torch.from_numpy(w.x_bits.view(np.int16)) for w in ws]
    ids = [torch.from_numpy(w.topk_idx) for w in ws]
    outs = [torch.empty((w0.S, w0.H), dtype=torch.int16) for _ in ws]
    workspace = torch.empty((moe.moe_run_host_workspace_bytes(shape, 3),), dtype=torch.uint8, device="cuda")
    err = np.full(3, -1, np.int32)
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_run_host(shape, xs, ids, None, outs, workspace, err_host=err)
    assert ei.value.status == moe.MOE_ERR_TOPK_OUT_OF_RANGE
    assert err.tolist() == [0, moe.MOE_ERR_TOPK_OUT_OF_RANGE, 0]
    # Batches without the bad id are still exact (pageable host buffers work too).
    np.testing.assert_array_equal(outs[2].numpy().view(np.uint16), _expected(ws[2], weights=False))


def test_fused_flag_falls_back_where_the_fused_kernel_does_not_apply():
    # P = 80 is beyond the fused kernel's limit: the separate calls run instead.
    ws = _batches(80, 160, 3, 64, 2, 2)
    got = _run(ws, fused=True)
    for w, g in zip(ws, got):
        np.testing.assert_array_equal(g, _expected(w))


def _expected_expert(w, weights=True):
    lay, nt, _ = oracle.run_all(w.P, w.E, w.C, w.expert_alignment, w.H, 0, w.x_bits, w.topk_idx, w.topk_weights)
    ex = oracle.notify_expert(w.P, w.E, w.topk_idx, nt["num_recv_tokens_per_expert"], nt["recv_expert_offset"])
    rows = int(ex["expert_part_base"][-1])
    dis = oracle.dispatch_expert(w.P, w.E, w.H, 0, w.x_bits, w.topk_idx, w.topk_weights, ex["slot_row"],
                                 ex["expert_part_base"], rows)
    ref = oracle.combine_expert(w.P, w.E, w.H, dis["arena"], oracle.slot_stride(w.H, 0), ex["expert_part_base"],
                                rows, ex["slot_row"], w.topk_idx, w.topk_weights if weights else None)
    return ref["out"]


def test_expert_major_batches_match_the_oracle():
    import torch

    ws = _batches(4, 16, 80, 256, 4, 3, mask_frac=0.1)
    w0 = ws[0]
    shape = moe.make_shape(w0.P, w0.E, w0.S, w0.K, w0.H, w0.C, w0.expert_alignment, 0)
    xs = [torch.from_numpy(w.x_bits.view(np.int16)).pin_memory() for w in ws]
    ids = [torch.from_numpy(w.topk_idx).pin_memory() for w in ws]
    wts = [torch.from_numpy(w.topk_weights).pin_memory() for w in ws]
    outs = [torch.empty((w0.S, w0.H), dtype=torch.int16).pin_memory() for _ in ws]
    workspace = torch.empty((moe.moe_run_host_workspace_bytes(shape, 3),), dtype=torch.uint8, device="cuda")
    moe.moe_run_host(shape, xs, ids, wts, outs, workspace, expert=True)
    for w, o in zip(ws, outs):
        np.testing.assert_array_equal(o.numpy().view(np.uint16), _expected_expert(w))


def test_no_tokens_runs_and_reports_no_error():
    import torch

    shape = moe.make_shape(4, 16, 0, 2, 64)
    empty_x = torch.empty((0, 64), dtype=torch.int16).pin_memory()
    empty_i = torch.empty((0, 2), dtype=torch.int32).pin_memory()
    out = torch.empty((0, 64), dtype=torch.int16).pin_memory()
    workspace = torch.empty((moe.moe_run_host_workspace_bytes(shape, 2),), dtype=torch.uint8, device="cuda")
    err = np.full(2, -1, np.int32)
    for fused in (False, True):
        moe.moe_run_host(shape, [empty_x] * 2, [empty_i] * 2, None, [out] * 2, workspace, fused=fused, err_host=err)
        assert (err == 0).all()
