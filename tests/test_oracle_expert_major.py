"""Pins for the oracle's expert-major receive layout (CPU only).

The layout copies each (token, k) slot to its expert's rows, in the order of
"HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 3.6 (dstExpertOffset +
curExpertCnt), and combines per slot in k order (section 7.8).
"""

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs
from tests.helpers import bf16_bits_to_f32, f32_to_bf16_bits_torch


def _tables(P, E, idx, A=1, C=4):
    lay = oracle.layout(P, E, idx)
    nt = oracle.notify(P, E, C, A, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    ex = oracle.notify_expert(P, E, idx, nt["num_recv_tokens_per_expert"], nt["recv_expert_offset"])
    return lay, nt, ex


def test_hand_worked_example():
    # P=2 ranks, E=4 experts (2 per rank), K=2, four tokens.
    idx = np.array([[1, 2], [1, 3], [0, 1], [-1, 2]], np.int32)
    _, _, ex = _tables(2, 4, idx)
    # expert 0: (2,0) | expert 1: (0,0) (1,0) (2,1) | expert 2: (0,1) (3,1) | expert 3: (1,1)
    assert ex["slot_row"].tolist() == [[1, 0], [2, 2], [0, 3], [-1, 1]]
    assert ex["expert_part_base"].tolist() == [0, 4, 7]
    # With expert_alignment 4 every expert segment starts on a multiple of 4.
    _, _, ex4 = _tables(2, 4, idx, A=4)
    assert ex4["slot_row"].tolist() == [[4, 0], [5, 4], [0, 6], [-1, 1]]
    assert ex4["expert_part_base"].tolist() == [0, 8, 16]


@pytest.mark.parametrize("name,T,A", [("tiny_p4_e16_h256", None, 1),
                                      ("p128_e256_t512_h7168_zipf", 20, 3),
                                      ("p32_e256_t128_h1024", 16, 8)])
def test_rows_follow_stable_sort_by_expert(name, T, A):
    w = inputs.workload(name, T=T, with_x=False)
    lay, nt, ex = _tables(w.P, w.E, w.topk_idx, A=A, C=w.C)
    idx = w.topk_idx.reshape(-1)
    sr = ex["slot_row"].reshape(-1)
    valid = (idx >= 0) & (idx < w.E)
    assert (sr[~valid] == -1).all()
    slots = np.nonzero(valid)[0]                       # (token, k) order
    order = slots[np.argsort(idx[slots], kind="stable")]
    e_sorted = idx[order]
    starts = np.searchsorted(e_sorted, np.arange(w.E))
    pos = np.arange(order.shape[0]) - starts[e_sorted]
    want = nt["recv_expert_offset"].reshape(-1)[e_sorted] + pos
    np.testing.assert_array_equal(sr[order], want)
    # Each expert's slots fit its aligned count; partitions hold the aligned totals.
    raw = np.bincount(idx[valid], minlength=w.E)
    assert (raw <= nt["num_recv_tokens_per_expert"].reshape(-1)).all()
    totals = nt["num_recv_tokens_per_expert"].sum(axis=1)
    np.testing.assert_array_equal(np.diff(ex["expert_part_base"]), totals)


def test_dispatch_and_combine_closed_forms():
    w = inputs.workload("tiny_p4_e16_h256")
    lay, nt, ex = _tables(w.P, w.E, w.topk_idx, C=w.C)
    rows = int(ex["expert_part_base"][-1])
    dis = oracle.dispatch_expert(w.P, w.E, w.H, 0, w.x_bits, w.topk_idx, w.topk_weights,
                                 ex["slot_row"], ex["expert_part_base"], rows)
    assert dis["err"] == 0
    epr = w.E // w.P
    stride = oracle.slot_stride(w.H, 0)
    triple_off = 2 * w.H + 32
    for g in range(w.S):
        for k in range(w.K):
            e = w.topk_idx[g, k]
            r = int(ex["expert_part_base"][e // epr] + ex["slot_row"][g, k])
            np.testing.assert_array_equal(dis["arena"][r, :2 * w.H].view(np.uint16), w.x_bits[g])
            assert dis["arena"][r, triple_off:triple_off + 12].view(np.int32).tolist() == [
                g // w.T, g % w.T, k]
            assert dis["recv_src_idx"][r] == g % w.T
            assert dis["recv_weight"][r] == w.topk_weights[g, k]
    # Unit weights, identity experts: out = bf16(x * K) (all K slots valid here).
    res = oracle.combine_expert(w.P, w.E, w.H, dis["arena"], stride, ex["expert_part_base"], rows,
                                ex["slot_row"], w.topk_idx, None)
    want = f32_to_bf16_bits_torch(bf16_bits_to_f32(w.x_bits) * np.float32(w.K) + np.float32(0))
    np.testing.assert_array_equal(res["out"], want)
    # Softmax weights summing to 1, identity experts: x back (-0 becomes +0).
    res = oracle.combine_expert(w.P, w.E, w.H, dis["arena"], stride, ex["expert_part_base"], rows,
                                ex["slot_row"], w.topk_idx, w.topk_weights)
    np.testing.assert_array_equal(
        res["out"], f32_to_bf16_bits_torch(bf16_bits_to_f32(w.x_bits) + np.float32(0)))


def _crafted(values, weights, experts, P=4, E=8, H=8):
    K = len(experts)
    idx = np.full((P, K), -1, np.int32)
    idx[0] = experts
    wts = np.zeros((P, K), np.float32)
    wts[0] = weights
    lay, nt, ex = _tables(P, E, idx, C=1)
    rows = int(ex["expert_part_base"][-1])
    y = np.zeros((rows, H), np.uint16)
    epr = E // P
    for k, v in enumerate(values):
        r = int(ex["expert_part_base"][experts[k] // epr] + ex["slot_row"][0, k])
        y[r] = f32_to_bf16_bits_torch(np.full(H, v, np.float32))
    res = oracle.combine_expert(P, E, H, y, 2 * H, ex["expert_part_base"], rows, ex["slot_row"], idx, wts)
    return bf16_bits_to_f32(res["out"][0])


def test_slots_reduced_in_k_order():
    # Two slots on the same rank (experts 0 and 1), one on rank 1: k order, not rank order.
    out = _crafted([2.0 ** 24, 1.0, -(2.0 ** 24)], [1, 1, 1], [0, 2, 1])
    assert (out == 0.0).all()


def test_slot_products_not_fused():
    Pv = np.float32(1.0 + 2 ** -7 + 2 ** -23)
    c1 = np.float32(1.0 + 2 ** -23)
    out = _crafted([-1.0, 1.0 + 2 ** -7], [Pv, c1], [3, 0])
    assert (out == 0.0).all() and not np.signbit(out).any()
