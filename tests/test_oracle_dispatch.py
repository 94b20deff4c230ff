"""Pins for the oracle's dispatch step, BF16 and int8 (CPU only)."""

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs
from tests.helpers import bf16_bits_to_f32


def _ceil(v, m):
    return (v + m - 1) // m * m


def _offsets(H, quant):
    elt = 1 if quant else 2
    scale_off = _ceil(H * elt, 32)
    return scale_off, scale_off + 32


def _numpy_quant(x_bits):
    """Dynamic int8 quantisation in numpy binary32 arithmetic."""
    xf = bf16_bits_to_f32(x_bits)
    amax = np.float32(np.abs(xf).max())
    scale = np.float32(amax / np.float32(127.0))
    if amax == 0:
        return np.zeros(xf.shape, np.int8), scale
    q = np.rint(xf / scale)  # float32 / float32 -> float32; rint is half-to-even
    return np.clip(q, -127, 127).astype(np.int8), scale


@pytest.mark.parametrize("quant", [0, 1])
def test_dispatch_roundtrip_tiny(quant):
    w = inputs.workload("tiny_p4_e16_h256")
    lay, nt, dis = oracle.run_all(w.P, w.E, w.C, 1, w.H, quant, w.x_bits, w.topk_idx,
                                  w.topk_weights)
    assert dis["err"] == 0
    arena = dis["arena"]
    P, E, T, K, H = w.P, w.E, w.T, w.K, w.H
    epr = E // P
    stride = oracle.slot_stride(H, quant)
    assert arena.shape[1] == stride
    scale_off, triple_off = _offsets(H, quant)
    rows_seen = 0
    for g in range(w.S):
        dests = np.nonzero(lay["is_token_in_rank"][g])[0]
        q_ref, s_ref = _numpy_quant(w.x_bits[g]) if quant else (None, None)
        for d in dests:
            row = int(nt["part_row_base"][d] + nt["send_head"][g, d])
            slot = arena[row]
            if quant:
                np.testing.assert_array_equal(slot[:H].view(np.int8), q_ref)
                assert slot[scale_off:scale_off + 4].view(np.float32)[0] == s_ref
            else:
                np.testing.assert_array_equal(slot[:2 * H].view(np.uint16), w.x_bits[g])
            ks = [k for k in range(K) if w.topk_idx[g, k] >= 0 and w.topk_idx[g, k] // epr == d]
            triple = slot[triple_off:triple_off + 12].view(np.int32).tolist()
            assert triple == [g // T, g % T, min(ks)]
            assert dis["recv_src_idx"][row] == g % T
            for k in range(K):
                if k in ks:
                    assert dis["recv_topk_idx"][row, k] == w.topk_idx[g, k] % epr
                    assert dis["recv_topk_weights"][row, k] == w.topk_weights[g, k]
                else:
                    assert dis["recv_topk_idx"][row, k] == -1
                    assert dis["recv_topk_weights"][row, k] == 0.0
            rows_seen += 1
    assert rows_seen == arena.shape[0] == int(nt["part_row_base"][-1])


def test_page_example_two_copies():
    """A token with Top-2 experts on ranks 0 and 3 lands in exactly two slots."""
    P, E, K, H = 4, 8, 2, 64
    idx = np.array([[1, 7], [-1, -1], [-1, -1], [-1, -1]], np.int32)
    x = (np.arange(4 * H, dtype=np.uint16).reshape(4, H) | 0x3F00)
    wts = np.full((4, K), 0.5, np.float32)
    lay, nt, dis = oracle.run_all(P, E, 16, 1, H, 0, x, idx, wts)
    assert dis["arena"].shape[0] == 2
    assert nt["part_row_base"].tolist() == [0, 1, 1, 1, 2]
    for r in range(2):
        np.testing.assert_array_equal(dis["arena"][r, :2 * H].view(np.uint16), x[0])


def test_quant_matches_numpy_binary32():
    w = inputs.workload("tiny_p4_e16_h256")
    for g in range(w.S):
        q, s = oracle.quantize_row(w.x_bits[g])
        q_ref, s_ref = _numpy_quant(w.x_bits[g])
        assert s == s_ref
        np.testing.assert_array_equal(q, q_ref)


def test_quant_bounds_and_extremes():
    w = inputs.make(1, 1, 64, 7168, 1, seed=3)
    for g in range(w.S):
        q, s = oracle.quantize_row(w.x_bits[g])
        xf = bf16_bits_to_f32(w.x_bits[g]).astype(np.float64)
        # Half a step, plus the binary32 rounding of x / scale (|x / scale| <= 127).
        err = np.abs(q.astype(np.float64) - xf / float(s))
        assert (err <= 0.5 + 128 * 2.0 ** -24).all()
        assert np.abs(q).max() == 127
        assert q[np.argmax(np.abs(xf))] in (127, -127)


def test_quant_ties_round_to_even_and_zero_row():
    # amax = 127 makes scale exactly 1.0, so q = rint(x) with ties to even.
    vals = np.array([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, -127.0, 126.5], np.float32)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert (bf16_bits_to_f32(bits) == vals).all()
    q, s = oracle.quantize_row(bits)
    assert s == np.float32(1.0)
    assert q.tolist() == [127, 2, 4, -2, 0, 2, 0, -127, 126]
    q0, s0 = oracle.quantize_row(np.zeros(32, np.uint16))
    assert s0 == 0.0 and (q0 == 0).all()


def test_capacity_overflow_is_reported_and_skipped():
    w = inputs.workload("tiny_p4_e16_h256")
    lay = oracle.layout(w.P, w.E, w.topk_idx)
    nt = oracle.notify(w.P, w.E, w.C, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    cap = int(nt["num_recv_tokens"].min()) - 1   # every partition one short at least
    prb = np.arange(w.P + 1, dtype=np.int64) * cap
    dis = oracle.dispatch(w.P, w.E, w.H, 0, w.x_bits, w.topk_idx, w.topk_weights,
                          nt["send_head"], prb, cap * w.P)
    assert dis["err"] == 3
    # Rows inside capacity are still written correctly.
    for d in range(w.P):
        g = int(np.nonzero(nt["send_head"][:, d] == 0)[0][0])
        np.testing.assert_array_equal(dis["arena"][d * cap, :2 * w.H].view(np.uint16), w.x_bits[g])


def test_token_subset_writes_only_those_rows():
    w = inputs.workload("tiny_p4_e16_h256")
    lay, nt, full = oracle.run_all(w.P, w.E, w.C, 1, w.H, 1, w.x_bits, w.topk_idx, w.topk_weights)
    toks = np.array([3, 77, 200], np.int64)
    rows = int(nt["part_row_base"][-1])
    sub = oracle.dispatch(w.P, w.E, w.H, 1, w.x_bits, w.topk_idx, w.topk_weights, nt["send_head"],
                          nt["part_row_base"], rows, tokens=toks)
    written = [int(nt["part_row_base"][d] + nt["send_head"][g, d])
               for g in toks for d in range(w.P) if nt["send_head"][g, d] >= 0]
    np.testing.assert_array_equal(sub["arena"][written], full["arena"][written])
    others = np.setdiff1d(np.arange(rows), written)
    assert (sub["arena"][others] == 0).all()


def _worst_tokens_case():
    """P=2 ranks, capacity 256 rows each; rank 0 receives 237 rows (the page's
    example), rank 1 receives 200."""
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "worst_tokens.json")) as f:
        gold = json.load(f)
    P, E, K, H, T = 2, 4, 1, 64, 256
    idx = np.full((P * T, K), -1, np.int32)
    idx[:gold["received"], 0] = np.arange(gold["received"]) % 2          # experts 0/1 -> rank 0
    idx[gold["received"]:gold["received"] + 200, 0] = 2                  # expert 2 -> rank 1
    rng = np.random.default_rng(0)
    x = (rng.integers(0, 1 << 15, size=(P * T, H)) | 0x3C00).astype(np.uint16)
    w = np.ones((P * T, K), np.float32)
    return gold, P, E, K, H, T, idx, x, w


def test_worst_tokens_padding_matches_page_example():
    gold, P, E, K, H, T, idx, x, w = _worst_tokens_case()
    cap = gold["capacity"]
    lay = oracle.layout(P, E, idx)
    nt = oracle.notify(P, E, 4, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    assert nt["num_recv_tokens"].tolist() == [gold["received"], 200]
    prb = np.arange(P + 1, dtype=np.int64) * cap
    dis = oracle.dispatch(P, E, H, 0, x, idx, w, nt["send_head"], prb, P * cap)
    assert dis["err"] == 0
    oracle.pad_partitions(P, K, H, 0, nt["num_recv_tokens"], prb, dis["arena"], dis["recv_src_idx"],
                          dis["recv_topk_idx"], dis["recv_topk_weights"])
    _, triple_off = _offsets(H, 0)
    pad = np.arange(gold["received"], cap)
    assert pad.shape[0] == gold["padding_rows"]
    assert (dis["arena"][pad, :2 * H] == 0).all()                       # x = 0
    assert (dis["recv_topk_weights"][pad] == 0).all()                   # weights = 0
    assert (dis["recv_topk_idx"][pad] == -1).all()                      # topk_idx = -1
    assert (dis["recv_src_idx"][pad] == -1).all()
    assert (dis["arena"][pad, triple_off:triple_off + 12].view(np.int32) == -1).all()
    # The 237 valid rows are untouched by the padding: row r holds token r's x.
    for r in range(gold["received"]):
        np.testing.assert_array_equal(dis["arena"][r, :2 * H].view(np.uint16), x[r])
    # Rank 1: 200 valid rows, 56 padding rows.
    assert (dis["recv_topk_idx"][cap + 200:2 * cap] == -1).all()
    assert (dis["recv_topk_idx"][cap:cap + 200] == 0).all()
