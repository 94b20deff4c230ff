"""Pins for the oracle's combine step and its bf16 conversion (CPU only)."""

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs
from tests.helpers import bf16_bits_to_f32, bf16_ulp_distance, f32_to_bf16_bits_torch


def _pipeline(w, quant=0):
    lay, nt, dis = oracle.run_all(w.P, w.E, w.C, 1, w.H, quant, w.x_bits, w.topk_idx,
                                  w.topk_weights)
    return lay, nt, dis


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(20000) * 1e30).astype(np.float32),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),   # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8,
                  -(1.0 + 2 ** -8)], np.float32),
    ])
    # Exact ties: low 16 bits = 0x8000.
    ties = ((rng.integers(0, 1 << 16, 5000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    vals = np.concatenate([vals, ties])
    np.testing.assert_array_equal(oracle.bf16_round(vals), f32_to_bf16_bits_torch(vals))


def test_unit_weights_identity_experts_closed_form():
    """NULL weights, y = dispatched x: out = bf16(x * n_distinct), exact in fp32."""
    for name, T in [("tiny_p4_e16_h256", None), ("p128_e256_t512_h7168_zipf", 4)]:
        w = inputs.workload(name, T=T)
        lay, nt, dis = _pipeline(w)
        rows = int(nt["part_row_base"][-1])
        stride = oracle.slot_stride(w.H, 0)
        res = oracle.combine(w.P, w.E, w.H, dis["arena"], stride, nt["part_row_base"], rows,
                             nt["send_head"], w.topk_idx, None)
        assert res["err"] == 0
        n = lay["is_token_in_rank"].sum(axis=1).astype(np.float32)
        # The accumulator starts at +0, so a -0 input comes back as +0.
        want = f32_to_bf16_bits_torch(bf16_bits_to_f32(w.x_bits) * n[:, None] + np.float32(0.0))
        np.testing.assert_array_equal(res["out"], want)


def test_softmax_weights_identity_experts_return_x():
    """Top-K weights summing to 1 with identity experts give back x."""
    w = inputs.workload("tiny_p4_e16_h256")
    lay, nt, dis = _pipeline(w)
    rows = int(nt["part_row_base"][-1])
    res = oracle.combine(w.P, w.E, w.H, dis["arena"], oracle.slot_stride(w.H, 0),
                         nt["part_row_base"], rows, nt["send_head"], w.topk_idx, w.topk_weights)
    assert bf16_ulp_distance(res["out"], w.x_bits).max() <= 1
    plus_zero = f32_to_bf16_bits_torch(bf16_bits_to_f32(w.x_bits) + np.float32(0.0))
    np.testing.assert_array_equal(res["out"], plus_zero)


def test_within_error_bound_of_binary64_sum():
    """Against the exact (binary64) weighted sum: error <= final rounding + the
    textbook bound for a recursive binary32 sum of n rounded products."""
    w = inputs.workload("p32_e256_t128_h1024", T=8)
    lay, nt, dis = _pipeline(w)
    rows = int(nt["part_row_base"][-1])
    stride = oracle.slot_stride(w.H, 0)
    # Non-identity expert outputs: random bf16 rows in the arena.
    rng = np.random.default_rng(2)
    y = dis["arena"].copy()
    rnd = f32_to_bf16_bits_torch(rng.standard_normal((rows, w.H)).astype(np.float32))
    y[:, :2 * w.H] = rnd.view(np.uint8).reshape(rows, 2 * w.H)
    res = oracle.combine(w.P, w.E, w.H, y, stride, nt["part_row_base"], rows, nt["send_head"],
                         w.topk_idx, w.topk_weights)
    epr = w.E // w.P
    ref = np.zeros((w.S, w.H), np.float64)
    mag = np.zeros((w.S, w.H), np.float64)
    n = np.zeros((w.S, 1), np.float64)
    for g in range(w.S):
        for d in range(w.P):
            sh = nt["send_head"][g, d]
            if sh < 0:
                continue
            c = sum(float(w.topk_weights[g, k]) for k in range(w.K)
                    if w.topk_idx[g, k] >= 0 and w.topk_idx[g, k] // epr == d)
            term = c * bf16_bits_to_f32(rnd[int(nt["part_row_base"][d]) + sh]).astype(np.float64)
            ref[g] += term
            mag[g] += np.abs(term)
            n[g] += 1
    got = bf16_bits_to_f32(res["out"]).astype(np.float64)
    bound = 2.0 ** -8 * np.abs(ref) + (2 * n + 2 * w.K + 2) * 2.0 ** -24 * mag + 1e-38
    assert (np.abs(got - ref) <= bound).all()
    # Away from cancellation the result is the correctly rounded value or a neighbour.
    want = f32_to_bf16_bits_torch(ref.astype(np.float32))
    far = np.abs(ref) > 0.25 * mag
    assert bf16_ulp_distance(res["out"], want)[far].max() <= 1


def test_single_rank_reduces_to_plain_scale():
    """P = 1: one row per token, out = bf16(c * y) with c the binary32 sum of weights."""
    w = inputs.make(1, 8, 32, 256, 4, seed=9)
    lay, nt, dis = _pipeline(w)
    rows = int(nt["part_row_base"][-1])
    assert rows == w.S
    res = oracle.combine(1, w.E, w.H, dis["arena"], oracle.slot_stride(w.H, 0),
                         nt["part_row_base"], rows, nt["send_head"], w.topk_idx, w.topk_weights)
    c = np.zeros(w.S, np.float32)
    for k in range(w.K):
        c = (c + w.topk_weights[:, k]).astype(np.float32)
    want = f32_to_bf16_bits_torch((c[:, None] * bf16_bits_to_f32(w.x_bits)).astype(np.float32))
    np.testing.assert_array_equal(res["out"], want)


def _crafted(rows_f32, weights, experts, P=4, E=4, H=8):
    """One token (plus masked padding tokens), arena rows given per rank."""
    K = len(experts)
    S = P
    idx = np.full((S, K), -1, np.int32)
    idx[0] = experts
    wts = np.zeros((S, K), np.float32)
    wts[0] = weights
    lay = oracle.layout(P, E, idx)
    nt = oracle.notify(P, E, 1, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    rows = int(nt["part_row_base"][-1])
    y = np.zeros((rows, H), np.uint16)
    for d, v in rows_f32.items():
        r = int(nt["part_row_base"][d] + nt["send_head"][0, d])
        y[r] = f32_to_bf16_bits_torch(np.full(H, v, np.float32))
        assert (bf16_bits_to_f32(y[r]) == np.float32(v)).all()
    res = oracle.combine(P, E, H, y, 2 * H, nt["part_row_base"], rows, nt["send_head"], idx, wts)
    return bf16_bits_to_f32(res["out"][0])


def test_ranks_reduced_in_ascending_order():
    # 2^24 + 1 rounds back to 2^24 in binary32; ascending order gives 0,
    # descending order would give 1.
    out = _crafted({0: 2.0 ** 24, 1: 1.0, 2: -(2.0 ** 24)}, [1.0, 1.0, 1.0], [0, 1, 2])
    assert (out == 0.0).all()


def test_multiply_and_add_rounded_separately():
    # c0 * y0 = -P exactly; c1 * y1 = P + 2^-30 rounds to P. Unfused: 0; fused: 2^-30.
    Pval = np.float32(1.0 + 2 ** -7 + 2 ** -23)
    c1 = np.float32(1.0 + 2 ** -23)
    assert np.float32(c1 * np.float32(1.0 + 2 ** -7)) == Pval
    out = _crafted({0: -1.0, 1: 1.0 + 2 ** -7}, [Pval, c1], [0, 1])
    assert (out == 0.0).all() and not np.signbit(out).any()


def test_weights_of_one_rank_summed_in_k_order():
    # Two slots on rank 1 (experts 2 and 3 with epr = 2... here P=2, E=4).
    P, E, H = 2, 4, 8
    idx = np.array([[2, 0, 3], [-1, -1, -1]], np.int32)
    wts = np.array([[0.25, 0.5, 0.125], [0, 0, 0]], np.float32)
    lay = oracle.layout(P, E, idx)
    nt = oracle.notify(P, E, 1, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    rows = int(nt["part_row_base"][-1])
    y = np.zeros((rows, H), np.uint16)
    y[int(nt["part_row_base"][0])] = f32_to_bf16_bits_torch(np.full(H, 2.0, np.float32))
    y[int(nt["part_row_base"][1])] = f32_to_bf16_bits_torch(np.full(H, 4.0, np.float32))
    res = oracle.combine(P, E, H, y, 2 * H, nt["part_row_base"], rows, nt["send_head"], idx, wts)
    # rank 0: c = 0.5 -> 1.0 ; rank 1: c = 0.25 + 0.125 -> 1.5 ; total 2.5
    assert (bf16_bits_to_f32(res["out"][0]) == 2.5).all()
    assert (res["out"][1] == 0).all()  # no destination -> +0


@pytest.mark.parametrize("quant", [0])
def test_out_of_range_rows_are_reported(quant):
    w = inputs.workload("tiny_p4_e16_h256")
    lay, nt, dis = _pipeline(w)
    rows = int(nt["part_row_base"][-1])
    res = oracle.combine(w.P, w.E, w.H, dis["arena"], oracle.slot_stride(w.H, 0),
                         nt["part_row_base"], rows - 5, nt["send_head"], w.topk_idx, None)
    assert res["err"] == 3
