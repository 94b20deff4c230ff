"""Pins for the oracle's layout and notify steps (CPU only).

Each check compares the oracle with something other than itself: the pages'
worked examples (tests/golden), brute-force enumeration written differently
from the oracle's loops, numpy's stable sort and array_split, and invariants.
"""

import json
import os

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs
from tests.helpers import channel_sizes, stable_receive_rows

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _routing(name, T=None, seed=0):
    return inputs.workload(name, with_x=False, T=T, seed=seed)


def _bruteforce_layout(P, E, topk_idx):
    """Membership test against each rank's block of experts (no division)."""
    S, K = topk_idx.shape
    T = S // P
    epr = E // P
    itr = np.zeros((S, P), np.uint8)
    for g in range(S):
        row = set(int(e) for e in topk_idx[g] if 0 <= e < E)
        for d in range(P):
            block = range(d * epr, (d + 1) * epr)
            itr[g, d] = 1 if any(e in row for e in block) else 0
    ntpr = itr.reshape(P, T, P).sum(axis=1).astype(np.int32)
    ntpe = np.zeros((P, E), np.int32)
    for s in range(P):
        v = topk_idx[s * T:(s + 1) * T].ravel()
        v = v[(v >= 0) & (v < E)]
        ntpe[s] = np.bincount(v, minlength=E)
    return itr, ntpr, ntpe


def test_slot_stride_matches_page():
    with open(os.path.join(GOLDEN, "slot_stride.json")) as f:
        gold = json.load(f)
    assert len(gold["cases"]) >= 4
    for case in gold["cases"]:
        assert case["H"] * (1 if case["quant"] else 2) == case["payload_bytes"]
        assert oracle.slot_stride(case["H"], case["quant"]) == case["stride"], case


def _example_idx(ex):
    P, K = ex["P"], ex["K"]
    if "topk_idx" in ex:
        idx = np.array(ex["topk_idx"], np.int32)
        return idx, {str(g): v for g, v in enumerate(ex["destinations"])}
    S = P  # one token per source rank
    idx = np.full((S, K), -1, np.int32)
    for g, row in ex["topk_idx_rows"].items():
        idx[int(g)] = row
    return idx, ex["destinations_rows"]


def test_route_examples_from_pages():
    with open(os.path.join(GOLDEN, "route_examples.json")) as f:
        gold = json.load(f)
    for ex in gold["examples"]:
        P, E = ex["P"], ex["E"]
        idx, dests = _example_idx(ex)
        lay = oracle.layout(P, E, idx)
        assert lay["err"] == 0
        for g, want in dests.items():
            got = np.nonzero(lay["is_token_in_rank"][int(g)])[0].tolist()
            assert got == want, (ex["citation"], g)
        # Tokens not listed go nowhere.
        listed = {int(g) for g in dests}
        for g in range(idx.shape[0]):
            if g not in listed:
                assert lay["is_token_in_rank"][g].sum() == 0
        nt = oracle.notify(P, E, 4, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                           lay["is_token_in_rank"])
        for d, toks in ex.get("segments", {}).items():
            d = int(d)
            col = nt["send_head"][:, d]
            got = [int(g) for g in np.argsort(np.where(col >= 0, col, 1 << 30), kind="stable")
                   if col[g] >= 0]
            assert got == toks
            assert sorted(col[col >= 0].tolist()) == list(range(len(toks)))
        # The page's example has 2 copies for the token that hits ranks 0 and 3.
        assert int(nt["part_row_base"][-1]) == sum(len(v) for v in dests.values())


@pytest.mark.parametrize("name", ["tiny_p4_e16_h256"])
def test_layout_bruteforce_tiny(name):
    w = _routing(name)
    itr, ntpr, ntpe = _bruteforce_layout(w.P, w.E, w.topk_idx)
    lay = oracle.layout(w.P, w.E, w.topk_idx)
    assert lay["err"] == 0
    np.testing.assert_array_equal(lay["is_token_in_rank"], itr)
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], ntpr)
    np.testing.assert_array_equal(lay["num_tokens_per_expert"], ntpe)


def test_layout_bruteforce_masked_and_duplicates():
    rng = np.random.default_rng(5)
    P, E, T, K = 8, 32, 24, 6
    idx = rng.integers(-1, E, size=(P * T, K)).astype(np.int32)  # duplicates and masks
    itr, ntpr, ntpe = _bruteforce_layout(P, E, idx)
    lay = oracle.layout(P, E, idx)
    np.testing.assert_array_equal(lay["is_token_in_rank"], itr)
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], ntpr)
    np.testing.assert_array_equal(lay["num_tokens_per_expert"], ntpe)


def test_layout_invariants_zipf():
    w = _routing("p128_e256_t512_h7168_zipf")
    lay = oracle.layout(w.P, w.E, w.topk_idx)
    itr = lay["is_token_in_rank"]
    P, T = w.P, w.T
    # Per-rank counts are the column sums of the token -> rank table.
    np.testing.assert_array_equal(lay["num_tokens_per_rank"], itr.reshape(P, T, P).sum(axis=1))
    # Per-expert counts add up to the valid slots of each source rank.
    valid = (w.topk_idx >= 0).reshape(P, T * w.K).sum(axis=1)
    np.testing.assert_array_equal(lay["num_tokens_per_expert"].sum(axis=1), valid)
    # Exactly 10% of the slots are masked.
    assert (w.topk_idx < 0).sum() == int(0.1 * w.S * w.K)
    # Packed bits agree with the byte table.
    bits = lay["is_token_in_rank_bits"]
    unpacked = np.unpackbits(bits.view(np.uint8), axis=1, bitorder="little")[:, :P]
    np.testing.assert_array_equal(unpacked, itr)
    # Zipf routing skews receive counts across ranks.
    recv = itr.sum(axis=0)
    assert recv.max() > 20 * max(1, recv.min())


def test_layout_out_of_range_is_reported_and_skipped():
    w = _routing("tiny_p4_e16_h256")
    bad = w.topk_idx.copy()
    bad[5, 1] = w.E + 3
    bad[17, 0] = 1 << 20
    lay_bad = oracle.layout(w.P, w.E, bad)
    masked = bad.copy()
    masked[masked >= w.E] = -1
    lay_ref = oracle.layout(w.P, w.E, masked)
    assert lay_bad["err"] == 2 and lay_ref["err"] == 0
    for k in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank"):
        np.testing.assert_array_equal(lay_bad[k], lay_ref[k])


def _check_notify(w, lay, nt, A):
    P, E, T, C = w.P, w.E, w.T, w.C
    itr = lay["is_token_in_rank"]
    # Receive order = stable sort of (token, rank) pairs by rank.
    np.testing.assert_array_equal(nt["send_head"], stable_receive_rows(itr))
    # Rank prefix: monotone down each column, last row = receive totals.
    rpm = nt["rank_prefix_matrix"]
    assert (np.diff(rpm, axis=0) >= 0).all()
    np.testing.assert_array_equal(rpm[-1], itr.sum(axis=0))
    np.testing.assert_array_equal(nt["num_recv_tokens"], itr.sum(axis=0))
    np.testing.assert_array_equal(np.diff(nt["part_row_base"]), nt["num_recv_tokens"])
    assert nt["part_row_base"][0] == 0
    # Channel prefix: numpy's array_split gives the channel boundaries.
    sizes = channel_sizes(T, C)
    bounds = np.concatenate([[0], np.cumsum(sizes)])
    cpm = nt["channel_prefix_matrix"]
    per_src = itr.reshape(P, T, P)
    for c in range(C):
        cnt = per_src[:, bounds[c]:bounds[c + 1], :].sum(axis=1)          # [s, d]
        prev = cpm[:, :, c - 1] if c else 0
        np.testing.assert_array_equal(cpm[:, :, c] - prev, cnt)
    np.testing.assert_array_equal(cpm[:, :, -1], lay["num_tokens_per_rank"])
    # recv_channel_prefix: the rows of channel (s, c) in d start there and are contiguous.
    rcpm = nt["recv_channel_prefix_matrix"]
    sh = nt["send_head"].reshape(P, T, P)
    for s in range(P):
        for c in range(C):
            blk = sh[s, bounds[c]:bounds[c + 1], :]
            for d in range(P):
                rows = blk[:, d][blk[:, d] >= 0]
                start = rcpm[d, s, c]
                np.testing.assert_array_equal(rows, np.arange(start, start + rows.shape[0]))
    # Per-expert receive counts, aligned; offsets are their exclusive scan.
    epr = E // P
    raw = lay["num_tokens_per_expert"].sum(axis=0).reshape(P, epr)
    aligned = -(-raw // A) * A
    np.testing.assert_array_equal(nt["num_recv_tokens_per_expert"], aligned)
    excl = np.cumsum(aligned, axis=1) - aligned
    np.testing.assert_array_equal(nt["recv_expert_offset"], excl)


@pytest.mark.parametrize("name,T,A", [
    ("tiny_p4_e16_h256", None, 1),
    ("tiny_p4_e16_h256", 13, 4),
    ("p32_e256_t128_h1024", None, 7),
    ("p128_e256_t512_h7168_zipf", 40, 1),
])
def test_notify_against_stable_sort_and_split(name, T, A):
    w = _routing(name, T=T)
    lay = oracle.layout(w.P, w.E, w.topk_idx)
    nt = oracle.notify(w.P, w.E, w.C, A, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    _check_notify(w, lay, nt, A)


def test_channel_split_page_rule():
    """Balanced split: first T % C channels take one extra token."""
    P, E, K = 1, 4, 1
    for T, C, want in [(10, 4, [3, 6, 8, 10]), (3, 5, [1, 2, 3, 3, 3]), (8, 1, [8])]:
        idx = np.zeros((T, K), np.int32)  # every token on rank 0
        lay = oracle.layout(P, E, idx)
        nt = oracle.notify(P, E, C, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                           lay["is_token_in_rank"])
        assert nt["channel_prefix_matrix"][0, 0].tolist() == want


def test_empty_input():
    P, E, K = 4, 16, 2
    idx = np.zeros((0, K), np.int32)
    lay = oracle.layout(P, E, idx)
    assert lay["num_tokens_per_rank"].sum() == 0 and lay["num_tokens_per_expert"].sum() == 0
    nt = oracle.notify(P, E, 16, 1, lay["num_tokens_per_rank"], lay["num_tokens_per_expert"],
                       lay["is_token_in_rank"])
    assert nt["part_row_base"].tolist() == [0] * (P + 1)
    assert nt["channel_prefix_matrix"].sum() == 0
