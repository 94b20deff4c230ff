"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact for layout, notify, dispatch payload / scale / triple and side
arrays; combine within 1 bf16 ulp of the oracle (and, since both sides round
each product and sum in binary32 in the same order, bit-exact as well).
"""

import numpy as np
import pytest

from combine_moe_layout_02_gb300 import inputs, moe
from tests import gpu_path as gp

pytestmark = pytest.mark.gpu


def _check_all(w, quant=0, weights=True, y_mode="identity", sample=None, seed=0):
    """Every table in full; dispatch and combine for all tokens (or a sample);
    and, the arena having been filled with canaries, no byte written outside
    the slot fields of the rows the routing sends (guard rows past the arena
    included)."""
    gpu = gp.run_gpu(w, quant=quant, weights=weights, y_mode=y_mode, canary=True, guard_rows=3)
    lay, nt = gp.oracle_tables(w)
    assert gpu["layout_err"] == 0 and gpu["dispatch_err"] == 0 and gpu["combine_err"] == 0
    gp.assert_tables_equal(gpu, lay, nt)
    gp.check_canaries(gpu, quant, w.H, np.arange(int(nt["part_row_base"][-1])))
    tokens = None
    if sample is not None and sample < w.S:
        rng = np.random.default_rng(seed)
        tokens = np.sort(rng.choice(w.S, size=sample, replace=False))
        tokens[0], tokens[-1] = 0, w.S - 1   # first and last token always in
        tokens = np.unique(tokens)
    gp.compare_dispatch(w, quant, gpu, nt, tokens=tokens)
    gp.compare_combine(w, gpu, nt, tokens=tokens, weights=weights)
    return gpu, lay, nt


# ---- small sizes: whole outputs compared, several tiles and a ragged tail ----

@pytest.mark.parametrize("quant", [0, 1])
def test_tiny(quant):
    w = inputs.workload("tiny_p4_e16_h256")
    _check_all(w, quant=quant, y_mode="int8expert" if quant else "identity")


@pytest.mark.parametrize("name,T", [
    ("p8_e256_t4096_h7168", 300),            # ragged against 256-token tiles and 16 channels
    ("p128_e256_t512_h7168_zipf", 9),        # skewed, masked, tiny channels
    ("p32_e256_t128_h1024", 128),
    ("p32_e256_t128_h2048", 37),
])
def test_reduced_workloads(name, T):
    w = inputs.workload(name, T=T)
    _check_all(w)


def test_reduced_int8_with_expert_stage():
    w = inputs.workload("p8_e256_t4096_h7168_int8", T=300)
    _check_all(w, quant=1, y_mode="int8expert")


def test_random_expert_rows_and_unit_weights():
    w = inputs.workload("p32_e256_t128_h1024", T=40)
    _check_all(w, y_mode="random")
    _check_all(w, y_mode="random", weights=False)


@pytest.mark.parametrize("P,E,T,K,H,C,A", [
    (1, 8, 333, 4, 64, 16, 1),        # one rank: every token goes to rank 0
    (3, 12, 50, 4, 136, 5, 3),        # P not a multiple of 4 (byte paths), odd C, alignment 3
    (5, 5, 77, 5, 8, 200, 1),         # one expert per rank, more channels than tokens, H = 8
    (1024, 1024, 2, 16, 64, 2, 1),    # maximum ranks and Top-K
    (16, 4096, 20, 8, 16384, 16, 8),  # maximum experts and hidden size
    (64, 128, 3, 1, 32, 1, 1),        # K = 1, one channel
    # notify's cluster kernel (more tokens than one CTA of a source rank holds):
    (6, 24, 1500, 4, 64, 7, 2),       # P not a multiple of 4 (byte flag loads), clusters of 16
    (8, 64, 1025, 8, 64, 300, 1),     # one token past the one-CTA limit (16 warps x 16 tokens x 4 steps)
    (130, 260, 40, 8, 64, 50, 1),     # 33 rank groups: two rank blocks per warp; fewer tokens than channels
    (64, 128, 1000, 4, 64, 1500, 1),  # 125 channel starts x 64 ranks per CTA, past the shared-memory buffer: written directly
])
def test_edge_shapes(P, E, T, K, H, C, A):
    w = inputs.make(P, E, T, H, K, seed=P + K, mask_frac=0.05, C=C, expert_alignment=A)
    _check_all(w)


def test_edge_shapes_int8():
    w = inputs.make(3, 12, 50, 16 * 9, 4, seed=3, C=5)
    _check_all(w, quant=1, y_mode="int8expert")


def test_empty_input():
    w = inputs.make(4, 16, 0, 256, 2)
    gpu = gp.run_gpu(w)
    assert gpu["layout_err"] == 0
    assert gpu["num_tokens_per_rank"].sum() == 0 and gpu["num_tokens_per_expert"].sum() == 0
    assert gpu["part_row_base"].tolist() == [0] * 5
    assert gpu["channel_prefix_matrix"].sum() == 0


def test_all_masked_and_duplicates():
    w = inputs.make(8, 64, 40, 128, 6, seed=4)
    idx = w.topk_idx.copy()
    idx[:13] = -1                      # tokens with no destination
    idx[20:, 1] = idx[20:, 0]          # duplicate expert ids inside a row
    w.topk_idx = idx
    gpu, lay, nt = _check_all(w)
    assert (gpu["out"][:13] == 0).all()  # +0 for tokens that went nowhere


def test_zero_rows_quantise_to_zero():
    w = inputs.make(4, 16, 32, 256, 2, seed=6)
    w.x_bits[5] = 0
    w.x_bits[9] = 0x8000   # all -0
    _check_all(w, quant=1, y_mode="int8expert")


def test_out_of_range_expert_ids():
    w = inputs.make(4, 16, 64, 64, 2, seed=8)
    bad = w.topk_idx.copy()
    bad[3, 0] = 16
    bad[100, 1] = 1 << 30
    gpu = gp.run_gpu(w, topk_idx=bad)
    assert gpu["layout_err"] == moe.MOE_ERR_TOPK_OUT_OF_RANGE
    masked = bad.copy()
    masked[masked >= 16] = -1
    lay, nt = gp.oracle_tables(w, topk_idx=masked)
    gp.assert_tables_equal(gpu, lay, nt)


def test_fixed_capacity_partitions():
    w = inputs.make(4, 16, 64, 128, 2, seed=10)
    lay, nt = gp.oracle_tables(w)
    cap = int(nt["num_recv_tokens"].max())
    prb = np.arange(w.P + 1, dtype=np.int64) * cap
    gpu = gp.run_gpu(w, arena_rows=cap * w.P, part_row_base=prb, canary=True, guard_rows=4)
    assert gpu["dispatch_err"] == 0 and gpu["combine_err"] == 0
    _, rows = gp.compare_dispatch(w, 0, gpu, nt, part_row_base=prb)
    gp.check_canaries(gpu, 0, w.H, rows)  # the gaps at the partitions' ends stay untouched
    nt_cap = dict(nt, part_row_base=prb)
    gp.compare_combine(w, gpu, nt_cap)


@pytest.mark.parametrize("quant", [0, 1])
def test_capacity_overflow_reported_without_stray_writes(quant):
    """Partitions too small for their rows: the overflow is reported, the rows
    that fit are exact, and no byte is written anywhere else -- not in the
    padding of written slots, not in rows past a partition's rows, not in
    the guard rows allocated past the arena the call was given."""
    w = inputs.make(4, 16, 64, 128, 2, seed=10)
    lay, nt = gp.oracle_tables(w)
    cap = int(nt["num_recv_tokens"].min()) - 2
    prb = np.arange(w.P + 1, dtype=np.int64) * cap
    gpu = gp.run_gpu(w, quant=quant, arena_rows=cap * w.P, part_row_base=prb, canary=True, guard_rows=5,
                     y_mode="int8expert" if quant else "identity")
    assert gpu["dispatch_err"] == moe.MOE_ERR_CAPACITY
    _, rows = gp.compare_dispatch(w, quant, gpu, nt, part_row_base=prb)
    gp.check_canaries(gpu, quant, w.H, rows)


def test_deterministic_repeat():
    w = inputs.workload("p128_e256_t512_h7168_zipf", T=16)
    gpu = gp.run_gpu(w, repeat=2)
    a, b = gpu["runs"]
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def test_invalid_arguments_rejected_on_host():
    import torch

    w = inputs.make(4, 16, 16, 64, 2)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H)
    buf = moe.Buffers(shape, "cuda")
    x = torch.from_numpy(w.x_bits.view(np.int16)).cuda()
    idx = torch.from_numpy(w.topk_idx).cuda()
    wts = torch.from_numpy(w.topk_weights).cuda()
    buf.layout(idx)
    buf.notify()
    xbig = torch.zeros(w.S * w.H + 8, dtype=torch.int16, device="cuda")
    misaligned = xbig.data_ptr() + 2
    with pytest.raises(moe.MoeError) as e:
        moe.moe_dispatch(shape, misaligned, idx, wts, buf.send_head, buf.part_row_base,
                         buf.recv_arena, buf.arena_rows, None, None, None, buf.err)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    bad = moe.make_shape(4, 18, 16, 2, 64)   # E % P != 0
    with pytest.raises(moe.MoeError):
        moe.moe_layout(bad, idx, buf.num_tokens_per_rank, buf.num_tokens_per_expert,
                       buf.is_token_in_rank, None, buf.err, buf.scratch)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.moe_layout(shape, idx, buf.num_tokens_per_rank, buf.num_tokens_per_expert,
                       buf.is_token_in_rank, None, buf.err, small)
    torch.cuda.synchronize()
    buf.dispatch(x, idx, wts)   # the context is still healthy
    torch.cuda.synchronize()


# ---- full sizes, launch configuration of the benchmark: sampled outputs ----

@pytest.mark.parametrize("weights", [True, False])
def test_combine_over_every_finite_bf16_value(weights):
    """Expert outputs drawn from every finite bf16 value (denormals, both
    zeros, the largest magnitudes, so sums can overflow to infinity): combine
    equals the oracle bit for bit, with softmax and with unit weights."""
    w = inputs.make(8, 64, 512, 1024, 8, seed=51, mask_frac=0.05)
    _check_all(w, weights=weights, y_mode="allbf16")


@pytest.mark.parametrize("pattern,weights", [("0x7f7f", False), ("0xff7f", False), ("0x0001", True),
                                             ("0x8001", True)])
def test_combine_overflow_and_denormal_sums(pattern, weights):
    """Every expert output the largest finite bf16 (unit weights: a token on two
    or more ranks sums to infinity) or the smallest denormal (softmax weights:
    denormal products and sums), either sign: combine equals the oracle."""
    w = inputs.make(8, 64, 64, 256, 8, seed=53, mask_frac=0.05)
    gpu, _, _ = _check_all(w, weights=weights, y_mode="fill:" + pattern)
    if pattern in ("0x7f7f", "0xff7f"):
        assert ((gpu["out"] & 0x7FFF) == 0x7F80).any()  # some sums overflowed


def test_combine_column_halves_with_odd_chunk_count():
    """Enough tokens that combine deals (token, column half) units at any
    occupancy; H = 72 is 9 chunks of 8, so the halves are 4 and 5 chunks."""
    w = inputs.make(4, 16, 50000, 72, 2, seed=21, mask_frac=0.05)
    _check_all(w, sample=2000)


@pytest.mark.parametrize("name,quant,y_mode", [
    ("p8_e256_t4096_h7168", 0, "identity"),
    ("p8_e256_t4096_h7168_int8", 1, "int8expert"),
    ("p128_e256_t512_h7168_zipf", 0, "identity"),
    ("p32_e256_t128_h7168", 0, "identity"),
    ("p32_e256_t128_h1024", 0, "identity"),
])
def test_full_size_every_row(name, quant, y_mode):
    """The bench's workloads at full size, in the bench's launch configuration:
    every table, every received row (payload, scale, triple, side arrays) and
    every combined token compared with the oracle element by element, and the
    canary check over the whole arena."""
    import torch

    import oracle

    w = inputs.workload(name)
    gpu = gp.run_gpu(w, quant=quant, y_mode=y_mode, canary=True, guard_rows=2)
    assert gpu["layout_err"] == 0 and gpu["dispatch_err"] == 0 and gpu["combine_err"] == 0
    lay, nt = gp.oracle_tables(w)
    gp.assert_tables_equal(gpu, lay, nt)
    buf = gpu["buf"]
    R = int(nt["part_row_base"][-1])
    assert R == int(lay["is_token_in_rank"].sum())
    ref = oracle.dispatch(w.P, w.E, w.H, quant, w.x_bits, w.topk_idx, w.topk_weights, nt["send_head"],
                          nt["part_row_base"], R)
    assert ref["err"] == 0
    pay, scale_off, triple_off = gp.offsets(w.H, quant)
    got = buf.recv_arena[:R].cpu().numpy()
    np.testing.assert_array_equal(got[:, :pay], ref["arena"][:, :pay], err_msg="payload")
    np.testing.assert_array_equal(got[:, triple_off:triple_off + 12], ref["arena"][:, triple_off:triple_off + 12],
                                  err_msg="triple")
    if quant:
        np.testing.assert_array_equal(got[:, scale_off:scale_off + 4], ref["arena"][:, scale_off:scale_off + 4],
                                      err_msg="scale")
    for k in ("recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        np.testing.assert_array_equal(getattr(buf, k)[:R].cpu().numpy(), ref[k][:R], err_msg=k)
    del got
    gp.check_canaries(gpu, quant, w.H, np.arange(R))
    # Combine over every token, on the y rows the GPU combine read.
    if y_mode == "identity":
        y, y_stride = ref["arena"], buf.stride  # equal to the GPU arena in every byte combine reads
    else:
        y, y_stride = gpu["y"][:R].cpu().numpy().view(np.uint8), 2 * w.H
    comb = oracle.combine(w.P, w.E, w.H, np.ascontiguousarray(y), y_stride, nt["part_row_base"], R,
                          nt["send_head"], w.topk_idx, w.topk_weights)
    np.testing.assert_array_equal(gpu["out"], comb["out"], err_msg="combine")
    if y_mode == "identity" and not (w.topk_idx < 0).any():
        # softmax weights with identity experts give x back within 1 ulp
        from tests.helpers import bf16_ulp_distance
        assert bf16_ulp_distance(gpu["out"], w.x_bits).max() <= 1
    del ref, comb
    torch.cuda.empty_cache()


def test_cached_dispatch_reuses_the_handle():
    """Same routing, new hidden rows: dispatch with the handle of the first
    pass (no layout / notify) equals a fresh dispatch of the new rows."""
    import torch

    w = inputs.workload("p32_e256_t128_h1024", T=33)
    gpu = gp.run_gpu(w)
    buf = gpu["buf"]
    lay, nt = gp.oracle_tables(w)
    w2 = inputs.workload("p32_e256_t128_h1024", T=33, seed=5)   # same shape, new x (and routing)
    w.x_bits = w2.x_bits
    x2 = torch.from_numpy(w.x_bits.view(np.int16)).cuda()
    idx = torch.from_numpy(w.topk_idx).cuda()
    wts = torch.from_numpy(w.topk_weights).cuda()
    buf.recv_arena.zero_()
    buf.dispatch(x2, idx, wts)
    out = torch.empty((w.S, w.H), dtype=torch.int16, device="cuda")
    buf.combine(out, idx, wts)
    torch.cuda.synchronize()
    assert int(buf.err[0].item()) == 0
    gp.compare_dispatch(w, 0, gpu, nt)
    gpu["out"] = out.cpu().numpy().view(np.uint16)
    gp.compare_combine(w, gpu, nt)


@pytest.mark.parametrize("quant", [0, 1])
def test_fixed_capacity_with_padding(quant):
    """num_worst_tokens form: fixed partitions, padding rows filled by
    moe_pad_partitions exactly as the oracle fills them."""
    import torch
    import oracle

    w = inputs.make(4, 16, 100, 256, 3, seed=12, mask_frac=0.2)
    lay, nt = gp.oracle_tables(w)
    cap = int(nt["num_recv_tokens"].max()) + 7
    prb = np.arange(w.P + 1, dtype=np.int64) * cap
    gpu = gp.run_gpu(w, quant=quant, arena_rows=cap * w.P, part_row_base=prb,
                     y_mode="int8expert" if quant else "identity")
    buf = gpu["buf"]
    buf.pad()
    torch.cuda.synchronize()
    ref = oracle.dispatch(w.P, w.E, w.H, quant, w.x_bits, w.topk_idx, w.topk_weights,
                          nt["send_head"], prb, cap * w.P)
    oracle.pad_partitions(w.P, w.K, w.H, quant, nt["num_recv_tokens"], prb, ref["arena"],
                          ref["recv_src_idx"], ref["recv_topk_idx"], ref["recv_topk_weights"])
    pay, scale_off, triple_off = gp.offsets(w.H, quant)
    g_arena = buf.recv_arena.cpu().numpy()
    np.testing.assert_array_equal(g_arena[:, :pay], ref["arena"][:, :pay])
    np.testing.assert_array_equal(g_arena[:, triple_off:triple_off + 12],
                                  ref["arena"][:, triple_off:triple_off + 12])
    if quant:
        np.testing.assert_array_equal(g_arena[:, scale_off:scale_off + 4],
                                      ref["arena"][:, scale_off:scale_off + 4])
    for k in ("recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        np.testing.assert_array_equal(getattr(buf, k).cpu().numpy(), ref[k], err_msg=k)


def test_int8_exact_ties_take_the_division_path():
    """Rows whose quotients x / scale are exact half-integers (scale = 1 and
    scale = 1/8): round-half-even must match the oracle's IEEE division bit
    for bit, also when the quotient is reached through the reciprocal."""
    w = inputs.make(2, 4, 8, 256, 2, seed=31)
    f = np.zeros((w.S, w.H), np.float32)
    ks = np.arange(-127, 127, dtype=np.float32)
    f[0, :ks.shape[0]] = ks + 0.5          # ties at scale 1 (amax 127 set below)
    f[0, -1] = 127.0
    f[1, :ks.shape[0]] = (2 * ks + 1) / 16  # ties at scale 1/8 (amax 15.875)
    f[1, -1] = -15.875
    rng = np.random.default_rng(4)
    # Odd multiples of 1/16 (bf16-exact); rows whose amax is 15.875 tie exactly.
    f[2:] = ((2 * rng.integers(-127, 127, size=(w.S - 2, w.H)) + 1) / 16).astype(np.float32)
    w.x_bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert ((w.x_bits.astype(np.uint32) << 16).view(np.float32) == f).all()
    _check_all(w, quant=1, y_mode="int8expert")


def test_int8_quantisation_over_every_bf16_value():
    """For 65 amax values spread over the whole bf16 range (denormal to the
    largest finite), rows that hold amax and every bf16 value of magnitude at
    most amax: each int8 byte and scale equals the oracle's (IEEE division,
    round half to even) -- the ties that bf16 ratios hit included."""
    H = 16384
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    rows = []
    for b in [(e << 7) | m for e in range(0, 255, 12) for m in (0, 0x2A, 0x7F)]:
        if b == 0:
            continue
        amax = (np.array([b], np.uint32) << 16).view(np.float32)[0]
        sel = bits[finite & (np.abs(vals) <= amax)].astype(np.uint16)
        for r0 in range(0, sel.shape[0], H - 1):
            row = np.zeros(H, np.uint16)
            row[0] = b
            chunk = sel[r0:r0 + H - 1]
            row[1:1 + chunk.shape[0]] = chunk
            rows.append(row)
    x = np.stack(rows)
    w = inputs.make(1, 1, x.shape[0], H, 1, seed=41, quant=1)
    w.x_bits = x
    _check_all(w, quant=1, y_mode="random")


@pytest.mark.parametrize("H", [16384, 1024])
def test_int8_ring_depths(H):
    """int8 dispatch with 32 KB rows (ring of one slot per consumer warp) and
    2 KB rows (two slots per consumer warp)."""
    w = inputs.make(4, 16, 40, H, 3, seed=H % 97, mask_frac=0.1)
    _check_all(w, quant=1, y_mode="int8expert")
