"""Parity of the expert-major path (moe_notify_expert / moe_dispatch_expert /
moe_combine_expert, through the C ABI) with the CPU oracle: slot rows and
partition bases, slot bytes and side arrays bit-exact; combine bit-exact (and
within the 1-ulp bar)."""

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs, moe
from tests import gpu_path as gp
from tests.helpers import bf16_ulp_distance

pytestmark = pytest.mark.gpu


def _run(w, quant=0, weights=True, y_mode="identity", sample=None, seed=0):
    import torch

    dev = torch.device("cuda", 0)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, quant)
    buf = moe.Buffers(shape, dev, side_arrays=False)
    x = torch.from_numpy(w.x_bits.view(np.int16)).to(dev)
    idx = torch.from_numpy(w.topk_idx).to(dev)
    wts = torch.from_numpy(w.topk_weights).to(dev)
    buf.err.zero_()
    buf.layout(idx)
    buf.notify()
    buf.notify_expert(idx)
    buf.expert_arena.zero_()
    buf.expert_src_idx.fill_(-7)
    buf.expert_weight.fill_(-7.0)
    buf.dispatch_expert(x, idx, wts)
    torch.cuda.synchronize()
    assert int(buf.err[0].item()) == 0
    lay, nt = gp.oracle_tables(w)
    ex = oracle.notify_expert(w.P, w.E, w.topk_idx, nt["num_recv_tokens_per_expert"],
                              nt["recv_expert_offset"])
    np.testing.assert_array_equal(buf.slot_row.cpu().numpy(), ex["slot_row"])
    np.testing.assert_array_equal(buf.expert_part_base.cpu().numpy(), ex["expert_part_base"])
    rows_total = int(ex["expert_part_base"][-1])

    tokens = np.arange(w.S)
    if sample is not None and sample < w.S:
        tokens = np.unique(np.concatenate([[0, w.S - 1], np.random.default_rng(seed).choice(
            w.S, size=sample, replace=False)]))
    ref = oracle.dispatch_expert(w.P, w.E, w.H, quant, w.x_bits, w.topk_idx, w.topk_weights,
                                 ex["slot_row"], ex["expert_part_base"], buf.expert_rows,
                                 tokens=None if sample is None else tokens,
                                 arena=np.zeros((buf.expert_rows, buf.stride), np.uint8))
    epr = w.E // w.P
    rows = []
    for g in tokens:
        for k in range(w.K):
            e = w.topk_idx[g, k]
            if 0 <= e < w.E:
                rows.append(int(ex["expert_part_base"][e // epr] + ex["slot_row"][g, k]))
    rows = np.array(sorted(rows), np.int64)
    pay, scale_off, triple_off = gp.offsets(w.H, quant)
    rt = torch.from_numpy(rows).to(dev)
    g_arena = buf.expert_arena.index_select(0, rt).cpu().numpy()
    r_arena = ref["arena"][rows]
    np.testing.assert_array_equal(g_arena[:, :pay], r_arena[:, :pay])
    np.testing.assert_array_equal(g_arena[:, triple_off:triple_off + 12], r_arena[:, triple_off:triple_off + 12])
    if quant:
        np.testing.assert_array_equal(g_arena[:, scale_off:scale_off + 4], r_arena[:, scale_off:scale_off + 4])
    np.testing.assert_array_equal(buf.expert_src_idx.index_select(0, rt).cpu().numpy(), ref["recv_src_idx"][rows])
    np.testing.assert_array_equal(buf.expert_weight.index_select(0, rt).cpu().numpy(), ref["recv_weight"][rows])

    # combine over y rows
    if y_mode == "identity":
        y, ystride = buf.expert_arena, buf.stride
    elif y_mode == "dequant":
        a = buf.expert_arena[:max(rows_total, 1)]
        q = a[:, :w.H].view(torch.int8).float()
        sc = a[:, scale_off:scale_off + 4].contiguous().view(torch.float32)
        y = (q * sc).to(torch.bfloat16).view(torch.int16).contiguous()
        ystride = 2 * w.H
    else:
        g_ = torch.Generator(device="cpu").manual_seed(77)
        y = torch.randn((buf.expert_rows, w.H), generator=g_).to(torch.bfloat16).view(torch.int16).to(dev)
        ystride = 2 * w.H
    out = torch.full((w.S, w.H), 0x5555, dtype=torch.int16, device=dev)
    y_rows = y.shape[0]
    moe.moe_combine_expert(shape, y, ystride, buf.expert_part_base, y_rows, buf.slot_row, idx,
                           wts if weights else None, out, buf.err)
    torch.cuda.synchronize()
    assert int(buf.err[0].item()) == 0
    yb = y.view(torch.uint8).reshape(y.shape[0], -1)[:, :2 * w.H].cpu().numpy()
    res = oracle.combine_expert(w.P, w.E, w.H, np.ascontiguousarray(yb), 2 * w.H, ex["expert_part_base"],
                                yb.shape[0], ex["slot_row"], w.topk_idx,
                                w.topk_weights if weights else None, tokens=tokens)
    got = out.cpu().numpy().view(np.uint16)[tokens]
    want = res["out"][tokens]
    assert bf16_ulp_distance(got, want).max() <= 1
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("quant", [0, 1])
def test_tiny_expert_major(quant):
    _run(inputs.workload("tiny_p4_e16_h256"), quant=quant, y_mode="dequant" if quant else "identity")


@pytest.mark.parametrize("name,T", [("p8_e256_t4096_h7168", 300), ("p128_e256_t512_h7168_zipf", 9),
                                    ("p32_e256_t128_h1024", 70)])
def test_reduced_expert_major(name, T):
    _run(inputs.workload(name, T=T))


def test_random_rows_unit_weights_alignment():
    w = inputs.make(8, 64, 50, 256, 6, seed=21, mask_frac=0.15, expert_alignment=8, C=3)
    _run(w, y_mode="random")
    _run(w, y_mode="random", weights=False)


@pytest.mark.parametrize("P,E,T,K,H", [(1, 8, 100, 3, 64), (1024, 1024, 2, 16, 64), (16, 4096, 20, 8, 512),
                                       (5, 5, 33, 5, 8)])
def test_expert_major_edge_shapes(P, E, T, K, H):
    _run(inputs.make(P, E, T, H, K, seed=P + E, mask_frac=0.05))


@pytest.mark.parametrize("name,quant", [("p8_e256_t4096_h7168", 0), ("p128_e256_t512_h7168_zipf", 0),
                                        ("p8_e256_t4096_h7168_int8", 1)])
def test_expert_major_full_size_sampled(name, quant):
    _run(inputs.workload(name), quant=quant, y_mode="dequant" if quant else "identity", sample=800)
