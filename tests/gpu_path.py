"""Test harness: run the CUDA path (through the C ABI) and the oracle on the
same seeded workload, and compare their outputs. Test infrastructure only."""

from __future__ import annotations

import numpy as np

import oracle
from combine_moe_layout_02_gb300 import moe


def ceil_to(v, m):
    return (v + m - 1) // m * m


def offsets(H, quant):
    elt = 1 if quant else 2
    scale_off = ceil_to(H * elt, 32)
    return H * elt, scale_off, scale_off + 32


def expert_stage_int8(arena, recv_topk_idx, rows, H):
    """Stand-in expert for int8 slots: y = bf16(f32(q) * scale * (1 + l / 64)),
    l = local expert of the slot's lowest k (from the triple)."""
    import torch

    _, scale_off, triple_off = offsets(H, 1)
    a = arena[:rows]
    q = a[:, :H].view(torch.int8).float()
    scale = a[:, scale_off:scale_off + 4].contiguous().view(torch.float32)
    kmin = a[:, triple_off + 8:triple_off + 12].contiguous().view(torch.int32).long()
    loc = torch.gather(recv_topk_idx[:rows].long(), 1, kmin.clamp(min=0)).float()
    y = (q * scale) * (1.0 + loc / 64.0)
    return y.to(torch.bfloat16).view(torch.int16).contiguous()


CANARY = 0xA5       # arena bytes before dispatch (canary runs)
SIDE_CANARY = -7    # side-array entries before dispatch


def run_gpu(w, quant=0, weights=True, arena_rows=None, part_row_base=None, y_mode="identity",
            topk_idx=None, repeat=1, canary=False, guard_rows=0):
    """Run layout -> notify -> dispatch -> combine on cuda:0; return numpy outputs.

    part_row_base (host int64 [P+1]) replaces notify's packed bases before
    dispatch (fixed-capacity partitions). y_mode: "identity" (combine reads the
    dispatch arena), "int8expert" (the stand-in expert above), "random"
    (fresh bf16 rows in a compact [rows, H] tensor), "allbf16" (every finite
    bf16 value, in a seeded order) or "fill:0x...." (one bf16 bit pattern).
    canary: the arena is filled with CANARY bytes (not zeros) before dispatch,
    so check_canaries can find stray writes. guard_rows: that many rows are
    allocated past the arena_rows the calls are given.
    """
    import torch

    dev = torch.device("cuda", 0)
    idx_np = w.topk_idx if topk_idx is None else topk_idx
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, quant)
    rows_given = moe.moe_max_recv_rows(shape) if arena_rows is None else arena_rows
    buf = moe.Buffers(shape, dev, arena_rows=rows_given + guard_rows)
    buf.arena_rows = rows_given  # the calls see only these rows; the guard rows follow
    x = torch.from_numpy(w.x_bits.view(np.int16)).to(dev)
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, np.int32)).to(dev)
    wts = torch.from_numpy(w.topk_weights).to(dev)
    out = torch.empty((w.S, w.H), dtype=torch.int16, device=dev)
    res = {}
    for _ in range(repeat):
        buf.err.zero_()
        buf.layout(idx)
        torch.cuda.synchronize()
        res["layout_err"] = int(buf.err[0].item())
        buf.notify()
        if part_row_base is not None:
            buf.part_row_base.copy_(torch.from_numpy(np.asarray(part_row_base, np.int64)))
        if canary:
            buf.recv_arena.fill_(CANARY)
        else:
            buf.recv_arena.zero_()
        buf.recv_src_idx.fill_(SIDE_CANARY)
        buf.recv_topk_idx.fill_(SIDE_CANARY)
        buf.recv_topk_weights.fill_(float(SIDE_CANARY))
        buf.dispatch(x, idx, wts)
        torch.cuda.synchronize()
        res["dispatch_err"] = int(buf.err[0].item())
        rows_total = int(buf.part_row_base[-1].item()) if part_row_base is None else buf.arena_rows
        if y_mode == "identity":
            y, y_stride, y_rows = buf.recv_arena, buf.stride, buf.arena_rows
        elif y_mode == "int8expert":
            y = expert_stage_int8(buf.recv_arena, buf.recv_topk_idx, buf.arena_rows, w.H)
            y_stride, y_rows = 2 * w.H, buf.arena_rows
        elif y_mode == "random":
            g = torch.Generator(device="cpu").manual_seed(1234)
            y = torch.randn((buf.arena_rows, w.H), generator=g).to(torch.bfloat16).view(torch.int16).to(dev)
            y_stride, y_rows = 2 * w.H, buf.arena_rows
        elif y_mode.startswith("fill:"):
            # every y element the given bf16 bit pattern, e.g. "fill:0x7f7f"
            pattern = np.int16(np.uint16(int(y_mode[5:], 16)).view(np.int16))
            y = torch.full((buf.arena_rows, w.H), int(pattern), dtype=torch.int16, device=dev)
            y_stride, y_rows = 2 * w.H, buf.arena_rows
        elif y_mode == "allbf16":
            # every finite bf16 value (denormals, zeros of both signs, the
            # largest magnitudes), repeated in a seeded order
            bits = np.arange(1 << 16, dtype=np.uint32)
            finite = bits[(bits & 0x7F80) != 0x7F80].astype(np.uint16)
            order = np.random.default_rng(77).permutation(np.resize(finite, buf.arena_rows * w.H))
            y = torch.from_numpy(order.reshape(buf.arena_rows, w.H).view(np.int16)).to(dev)
            y_stride, y_rows = 2 * w.H, buf.arena_rows
        else:
            raise ValueError(y_mode)
        out.fill_(0x5555)
        moe.moe_combine(shape, y, y_stride, buf.part_row_base, y_rows, buf.send_head, idx,
                        wts if weights else None, out, buf.err)
        torch.cuda.synchronize()
        res["combine_err"] = int(buf.err[0].item())
        rep = dict(
            num_tokens_per_rank=buf.num_tokens_per_rank.cpu().numpy(),
            num_tokens_per_expert=buf.num_tokens_per_expert.cpu().numpy(),
            is_token_in_rank=buf.is_token_in_rank.cpu().numpy(),
            is_token_in_rank_bits=buf.is_token_in_rank_bits.cpu().numpy().view(np.uint32),
            rank_prefix_matrix=buf.rank_prefix_matrix.cpu().numpy(),
            channel_prefix_matrix=buf.channel_prefix_matrix.cpu().numpy(),
            recv_channel_prefix_matrix=buf.recv_channel_prefix_matrix.cpu().numpy(),
            num_recv_tokens=buf.num_recv_tokens.cpu().numpy(),
            num_recv_tokens_per_expert=buf.num_recv_tokens_per_expert.cpu().numpy(),
            recv_expert_offset=buf.recv_expert_offset.cpu().numpy(),
            send_head=buf.send_head.cpu().numpy(),
            part_row_base=buf.part_row_base.cpu().numpy(),
            out=out.cpu().numpy().view(np.uint16),
        )
        res.setdefault("runs", []).append(rep)
        res.update(rep)
    res["buf"] = buf
    res["y"] = y
    res["y_stride"] = y_stride
    res["y_rows"] = y_rows
    res["rows_total"] = rows_total
    return res


def oracle_tables(w, topk_idx=None):
    idx = w.topk_idx if topk_idx is None else topk_idx
    lay = oracle.layout(w.P, w.E, idx)
    nt = oracle.notify(w.P, w.E, w.C, w.expert_alignment, lay["num_tokens_per_rank"],
                       lay["num_tokens_per_expert"], lay["is_token_in_rank"])
    return lay, nt


LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank",
               "is_token_in_rank_bits")
NOTIFY_KEYS = ("rank_prefix_matrix", "channel_prefix_matrix", "recv_channel_prefix_matrix",
               "num_recv_tokens", "num_recv_tokens_per_expert", "recv_expert_offset", "send_head",
               "part_row_base")


def assert_tables_equal(gpu, lay, nt):
    for k in LAYOUT_KEYS:
        np.testing.assert_array_equal(gpu[k], lay[k], err_msg=k)
    for k in NOTIFY_KEYS:
        np.testing.assert_array_equal(gpu[k], nt[k], err_msg=k)


def rows_of(tokens, send_head, part_row_base, arena_rows):
    """Arena rows written for the given tokens (rows outside their partition
    or the arena are skipped by both sides and left out)."""
    rows = []
    for g in tokens:
        for d in np.nonzero(send_head[g] >= 0)[0]:
            sh = int(send_head[g, d])
            r = int(part_row_base[d]) + sh
            if sh < part_row_base[d + 1] - part_row_base[d] and r < arena_rows:
                rows.append(r)
    return np.array(sorted(rows), np.int64)


def compare_dispatch(w, quant, gpu, nt, tokens=None, part_row_base=None):
    """Compare the defined bytes of every written slot and the side arrays."""
    import torch

    buf = gpu["buf"]
    prb = nt["part_row_base"] if part_row_base is None else np.asarray(part_row_base, np.int64)
    arena_rows = buf.arena_rows
    tok = None if tokens is None else np.asarray(tokens, np.int64)
    ref = oracle.dispatch(w.P, w.E, w.H, quant, w.x_bits, w.topk_idx, w.topk_weights,
                          nt["send_head"], prb, arena_rows, tokens=tok,
                          arena=np.zeros((arena_rows, buf.stride), np.uint8))
    rows = rows_of(range(w.S) if tok is None else tok, nt["send_head"], prb, arena_rows)
    pay, scale_off, triple_off = offsets(w.H, quant)
    rows_t = torch.from_numpy(rows).to(buf.recv_arena.device)
    g_arena = buf.recv_arena.index_select(0, rows_t).cpu().numpy()
    r_arena = ref["arena"][rows]
    np.testing.assert_array_equal(g_arena[:, :pay], r_arena[:, :pay], err_msg="payload")
    np.testing.assert_array_equal(g_arena[:, triple_off:triple_off + 12],
                                  r_arena[:, triple_off:triple_off + 12], err_msg="triple")
    if quant:
        np.testing.assert_array_equal(g_arena[:, scale_off:scale_off + 4],
                                      r_arena[:, scale_off:scale_off + 4], err_msg="scale")
    for k in ("recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        g = getattr(buf, k).index_select(0, rows_t).cpu().numpy()
        np.testing.assert_array_equal(g, ref[k][rows], err_msg=k)
    return ref["err"], rows


def compact_y(gpu, tokens, send_head, part_row_base, H):
    """Gather the y rows the sampled tokens read into a small packed arena."""
    import torch

    P = send_head.shape[1]
    y = gpu["y"]
    y_stride = gpu["y_stride"]
    per_d = [[] for _ in range(P)]
    for g in tokens:
        for d in np.nonzero(send_head[g] >= 0)[0]:
            per_d[d].append((g, int(part_row_base[d] + send_head[g, d])))
    sh2 = np.full_like(send_head, -1)
    prb2 = np.zeros(P + 1, np.int64)
    src_rows = []
    for d in range(P):
        prb2[d + 1] = prb2[d] + len(per_d[d])
        for j, (g, r) in enumerate(per_d[d]):
            sh2[g, d] = j
            src_rows.append(r)
    rows_t = torch.tensor(src_rows, dtype=torch.int64, device=y.device)
    flat = y.view(torch.uint8).reshape(y.shape[0], -1)[:, :2 * H] if y.dtype != torch.uint8 else y[:, :2 * H]
    ys = flat.index_select(0, rows_t).cpu().numpy() if len(src_rows) else np.zeros((0, 2 * H), np.uint8)
    return np.ascontiguousarray(ys), 2 * H, sh2, prb2


def compare_combine(w, gpu, nt, tokens=None, weights=True):
    """Oracle combine over the same y rows; bit-exact check plus the 1-ulp bar."""
    from tests.helpers import bf16_ulp_distance

    tok = np.arange(w.S) if tokens is None else np.asarray(tokens, np.int64)
    ys, ystride, sh2, prb2 = compact_y(gpu, tok, nt["send_head"], nt["part_row_base"], w.H)
    ref = oracle.combine(w.P, w.E, w.H, ys, ystride, prb2, int(prb2[-1]), sh2, w.topk_idx,
                         w.topk_weights if weights else None, tokens=tok)
    got = gpu["out"][tok]
    want = ref["out"][tok]
    dist = bf16_ulp_distance(got, want)
    assert dist.max() <= 1, f"combine beyond 1 bf16 ulp: max {dist.max()}"
    np.testing.assert_array_equal(got, want, err_msg="combine bits")


def check_canaries(gpu, quant, H, written_rows):
    """Stray-write check after a canary run (run_gpu(..., canary=True)): in
    every written row each byte outside the fields the slot format defines
    (payload; the scale block, int8 only; the triple block) still holds the
    canary, the defined blocks' padding is zero, and every other row of the
    allocation -- guard rows past arena_rows included -- and every side-array
    entry of an unwritten row still hold their canaries. Element-wise, on the
    device."""
    import torch

    buf = gpu["buf"]
    A = buf.recv_arena
    dev = A.device
    n_alloc = A.shape[0]
    pay, scale_off, triple_off = offsets(H, quant)
    written = torch.zeros(n_alloc, dtype=torch.bool, device=dev)
    if len(written_rows):
        written[torch.as_tensor(np.asarray(written_rows, np.int64), device=dev)] = True
    Wr = A[written]
    c = CANARY
    assert bool((Wr[:, pay:scale_off] == c).all()), "bytes between the payload and the scale block"
    if quant:
        assert bool((Wr[:, scale_off + 4:scale_off + 32] == 0).all()), "scale block padding"
    else:
        assert bool((Wr[:, scale_off:scale_off + 32] == c).all()), "bf16 slots leave the scale block alone"
    assert bool((Wr[:, triple_off + 12:triple_off + 32] == 0).all()), "triple block padding"
    assert bool((Wr[:, triple_off + 32:] == c).all()), "slot padding after the triple block"
    assert bool((A[~written] == c).all()), "rows nothing was sent to"
    for name in ("recv_src_idx", "recv_topk_idx", "recv_topk_weights"):
        t = getattr(buf, name)
        if t is None:
            continue
        assert bool((t[~written] == SIDE_CANARY).all()), name
