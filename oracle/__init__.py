"""CPU oracle for the MoE dispatch/combine hot path -- test infrastructure.

Only the tests, the smoke check and the CPU-baseline leg of the benchmark
import this package. It wraps ``moe_oracle.cpp`` (plain single-threaded C++,
built with ``-O2 -ffp-contract=off``) through ctypes and numpy. It shares no
code with the CUDA library in ``combine_moe_layout_02_gb300``; the two only see
the same seeded inputs.

What each function computes, and the page passage it follows, is stated in
``moe_oracle.cpp``. Parity status: every function here is pinned by the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py`` (brute force on small
inputs, invariants, closed forms, and the pages' worked examples under
``tests/golden/``).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (g++, -O2, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.oracle_slot_stride.restype = i64
    lib.oracle_slot_stride.argtypes = [i32, i32]
    lib.oracle_layout.restype = i32
    lib.oracle_layout.argtypes = [i32, i32, i64, i32, vp, vp, vp, vp, vp]
    lib.oracle_notify.restype = None
    lib.oracle_notify.argtypes = [i32, i32, i64, i32, i32, vp, vp, vp,
                                  vp, vp, vp, vp, vp, vp, vp, vp]
    lib.oracle_quantize_row.restype = ctypes.c_float
    lib.oracle_quantize_row.argtypes = [i32, vp, vp]
    lib.oracle_dispatch.restype = i32
    lib.oracle_dispatch.argtypes = [i32, i32, i64, i32, i32, i32, vp, vp, vp, vp, vp,
                                    vp, i64, vp, vp, vp, vp, i64]
    lib.oracle_combine.restype = i32
    lib.oracle_combine.argtypes = [i32, i32, i64, i32, i32, vp, i64, vp, i64, vp, vp,
                                   vp, vp, vp, i64]
    lib.oracle_notify_expert.restype = None
    lib.oracle_notify_expert.argtypes = [i32, i32, i64, i32, vp, vp, vp, vp, vp]
    lib.oracle_dispatch_expert.restype = i32
    lib.oracle_dispatch_expert.argtypes = [i32, i32, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, i64,
                                           vp, vp, vp, i64]
    lib.oracle_combine_expert.restype = i32
    lib.oracle_combine_expert.argtypes = [i32, i32, i64, i32, i32, vp, i64, vp, i64, vp, vp, vp, vp,
                                          vp, i64]
    lib.oracle_pad_partitions.restype = None
    lib.oracle_pad_partitions.argtypes = [i32, i32, i32, i32, vp, vp, vp, i64, vp, vp, vp]
    lib.oracle_bf16_round.restype = None
    lib.oracle_bf16_round.argtypes = [vp, vp, i64]
    _lib = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def slot_stride(H: int, quant: int) -> int:
    """Bytes per receive slot ("HCCL Window 模式 (Non-SHMEM) 代码深度剖析", section 8.2)."""
    return int(_load().oracle_slot_stride(int(H), int(quant)))


def layout(P: int, E: int, topk_idx: np.ndarray) -> dict:
    topk_idx = _c(topk_idx, np.int32)
    S, K = topk_idx.shape
    W = (P + 31) // 32
    out = dict(
        num_tokens_per_rank=np.empty((P, P), np.int32),
        num_tokens_per_expert=np.empty((P, E), np.int32),
        is_token_in_rank=np.empty((S, P), np.uint8),
        is_token_in_rank_bits=np.empty((S, W), np.uint32),
    )
    err = _load().oracle_layout(P, E, S, K, _p(topk_idx), _p(out["num_tokens_per_rank"]),
                                _p(out["num_tokens_per_expert"]), _p(out["is_token_in_rank"]),
                                _p(out["is_token_in_rank_bits"]))
    out["err"] = int(err)
    return out


def notify(P: int, E: int, C: int, expert_alignment: int, num_tokens_per_rank: np.ndarray,
           num_tokens_per_expert: np.ndarray, is_token_in_rank: np.ndarray) -> dict:
    ntpr = _c(num_tokens_per_rank, np.int32)
    ntpe = _c(num_tokens_per_expert, np.int32)
    itr = _c(is_token_in_rank, np.uint8)
    S = itr.shape[0]
    epr = E // P
    out = dict(
        rank_prefix_matrix=np.empty((P, P), np.int32),
        channel_prefix_matrix=np.empty((P, P, C), np.int32),
        recv_channel_prefix_matrix=np.empty((P, P, C), np.int32),
        num_recv_tokens=np.empty((P,), np.int32),
        num_recv_tokens_per_expert=np.empty((P, epr), np.int32),
        recv_expert_offset=np.empty((P, epr), np.int32),
        send_head=np.empty((S, P), np.int32),
        part_row_base=np.empty((P + 1,), np.int64),
    )
    _load().oracle_notify(P, E, S, C, expert_alignment, _p(ntpr), _p(ntpe), _p(itr),
                          _p(out["rank_prefix_matrix"]), _p(out["channel_prefix_matrix"]),
                          _p(out["recv_channel_prefix_matrix"]), _p(out["num_recv_tokens"]),
                          _p(out["num_recv_tokens_per_expert"]), _p(out["recv_expert_offset"]),
                          _p(out["send_head"]), _p(out["part_row_base"]))
    return out


def quantize_row(x_row_bits: np.ndarray):
    """Dynamic int8 quantisation of one bf16 row (given as uint16 bits)."""
    x_row_bits = _c(x_row_bits, np.uint16)
    q = np.empty(x_row_bits.shape[0], np.int8)
    scale = _load().oracle_quantize_row(int(x_row_bits.shape[0]), _p(x_row_bits), _p(q))
    return q, np.float32(scale)


def dispatch(P: int, E: int, H: int, quant: int, x_bits: np.ndarray, topk_idx: np.ndarray,
             topk_weights: np.ndarray, send_head: np.ndarray, part_row_base: np.ndarray,
             arena_rows: int, tokens: np.ndarray | None = None, arena: np.ndarray | None = None,
             side: bool = True) -> dict:
    """Run the dispatch oracle.

    ``arena`` (uint8 [arena_rows, stride]) is allocated with ``np.zeros`` when not
    given. With ``tokens`` only the rows of those tokens are written.
    """
    x_bits = _c(x_bits, np.uint16)
    topk_idx = _c(topk_idx, np.int32)
    topk_weights = _c(topk_weights, np.float32)
    send_head = _c(send_head, np.int32)
    prb = _c(part_row_base, np.int64)
    S, K = topk_idx.shape
    stride = slot_stride(H, quant)
    if arena is None:
        arena = np.zeros((arena_rows, stride), np.uint8)
    assert arena.flags.c_contiguous and arena.dtype == np.uint8 and arena.size >= arena_rows * stride
    out = dict(arena=arena)
    if side:
        out["recv_src_idx"] = np.full((arena_rows,), -7, np.int32)
        out["recv_topk_idx"] = np.full((arena_rows, K), -7, np.int32)
        out["recv_topk_weights"] = np.full((arena_rows, K), -7.0, np.float32)
    tok = None if tokens is None else _c(tokens, np.int64)
    err = _load().oracle_dispatch(
        P, E, S, K, H, quant, _p(x_bits), _p(topk_idx), _p(topk_weights), _p(send_head),
        _p(prb), _p(arena), int(arena_rows),
        _p(out.get("recv_src_idx")), _p(out.get("recv_topk_idx")), _p(out.get("recv_topk_weights")),
        _p(tok), 0 if tok is None else int(tok.shape[0]))
    out["err"] = int(err)
    return out


def _check_rows(y: np.ndarray, y_row_stride: int, arena_rows: int, H: int) -> None:
    """The C oracle reads ``arena_rows`` rows of ``2*H`` bytes ``y_row_stride``
    apart from ``y``; refuse a ``y`` that does not hold them."""
    if y_row_stride < 2 * H:
        raise ValueError(f"y_row_stride {y_row_stride} < 2*H = {2 * H}")
    if arena_rows > 0 and y.size < (arena_rows - 1) * y_row_stride + 2 * H:
        raise ValueError(f"y holds {y.size} bytes, fewer than {arena_rows} rows of stride {y_row_stride}")


def combine(P: int, E: int, H: int, y: np.ndarray, y_row_stride: int, part_row_base: np.ndarray,
            arena_rows: int, send_head: np.ndarray, topk_idx: np.ndarray,
            topk_weights: np.ndarray | None, tokens: np.ndarray | None = None) -> dict:
    """Run the combine oracle; ``y`` is the raw byte arena (rows y_row_stride apart)."""
    y = np.ascontiguousarray(y).view(np.uint8)
    _check_rows(y, y_row_stride, arena_rows, H)
    send_head = _c(send_head, np.int32)
    topk_idx = _c(topk_idx, np.int32)
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    prb = _c(part_row_base, np.int64)
    S, K = topk_idx.shape
    out = np.zeros((S, H), np.uint16)
    tok = None if tokens is None else _c(tokens, np.int64)
    err = _load().oracle_combine(P, E, S, K, H, _p(y), int(y_row_stride), _p(prb), int(arena_rows),
                                 _p(send_head), _p(topk_idx), _p(w), _p(out),
                                 _p(tok), 0 if tok is None else int(tok.shape[0]))
    return dict(out=out, err=int(err))


def notify_expert(P: int, E: int, topk_idx: np.ndarray, num_recv_tokens_per_expert: np.ndarray,
                  recv_expert_offset: np.ndarray) -> dict:
    """Expert-major receive rows of every (token, k) slot and the partition bases."""
    idx = _c(topk_idx, np.int32)
    S, K = idx.shape
    out = dict(slot_row=np.empty((S, K), np.int32), expert_part_base=np.empty((P + 1,), np.int64))
    _load().oracle_notify_expert(P, E, S, K, _p(idx), _p(_c(num_recv_tokens_per_expert, np.int32)),
                                 _p(_c(recv_expert_offset, np.int32)), _p(out["slot_row"]),
                                 _p(out["expert_part_base"]))
    return out


def dispatch_expert(P: int, E: int, H: int, quant: int, x_bits, topk_idx, topk_weights, slot_row,
                    expert_part_base, arena_rows: int, tokens=None, arena=None) -> dict:
    x_bits = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int32)
    S, K = idx.shape
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    stride = slot_stride(H, quant)
    if arena is None:
        arena = np.zeros((arena_rows, stride), np.uint8)
    out = dict(arena=arena, recv_src_idx=np.full((arena_rows,), -7, np.int32),
               recv_weight=np.full((arena_rows,), -7.0, np.float32))
    tok = None if tokens is None else _c(tokens, np.int64)
    err = _load().oracle_dispatch_expert(
        P, E, S, K, H, quant, _p(x_bits), _p(idx), _p(w), _p(_c(slot_row, np.int32)),
        _p(_c(expert_part_base, np.int64)), _p(arena), int(arena_rows), _p(out["recv_src_idx"]),
        _p(out["recv_weight"]), _p(tok), 0 if tok is None else int(tok.shape[0]))
    out["err"] = int(err)
    return out


def combine_expert(P: int, E: int, H: int, y, y_row_stride: int, expert_part_base, arena_rows: int,
                   slot_row, topk_idx, topk_weights, tokens=None) -> dict:
    y = np.ascontiguousarray(y).view(np.uint8)
    _check_rows(y, y_row_stride, arena_rows, H)
    idx = _c(topk_idx, np.int32)
    S, K = idx.shape
    w = None if topk_weights is None else _c(topk_weights, np.float32)
    out = np.zeros((S, H), np.uint16)
    tok = None if tokens is None else _c(tokens, np.int64)
    err = _load().oracle_combine_expert(P, E, S, K, H, _p(y), int(y_row_stride),
                                        _p(_c(expert_part_base, np.int64)), int(arena_rows),
                                        _p(_c(slot_row, np.int32)), _p(idx), _p(w), _p(out), _p(tok),
                                        0 if tok is None else int(tok.shape[0]))
    return dict(out=out, err=int(err))


def pad_partitions(P: int, K: int, H: int, quant: int, num_recv_tokens: np.ndarray,
                   part_row_base: np.ndarray, arena: np.ndarray, recv_src_idx=None,
                   recv_topk_idx=None, recv_topk_weights=None) -> None:
    """Fill the padding rows of fixed-length partitions in place."""
    nrt = _c(num_recv_tokens, np.int32)
    prb = _c(part_row_base, np.int64)
    assert arena.flags.c_contiguous and arena.dtype == np.uint8
    rows = arena.shape[0]
    for a, dt in ((recv_src_idx, np.int32), (recv_topk_idx, np.int32), (recv_topk_weights, np.float32)):
        assert a is None or (a.flags.c_contiguous and a.dtype == dt)
    _load().oracle_pad_partitions(P, K, H, quant, _p(nrt), _p(prb), _p(arena), int(rows),
                                  _p(recv_src_idx), _p(recv_topk_idx), _p(recv_topk_weights))


def bf16_round(values: np.ndarray) -> np.ndarray:
    """The oracle's binary32 -> bfloat16 (RNE) conversion, as uint16 bits."""
    v = _c(values, np.float32).ravel()
    out = np.empty(v.shape, np.uint16)
    _load().oracle_bf16_round(_p(v), _p(out), int(v.shape[0]))
    return out.reshape(np.shape(values))


def run_all(P, E, C, expert_alignment, H, quant, x_bits, topk_idx, topk_weights):
    """Layout -> notify -> dispatch (packed partitions) for small cases."""
    lay = layout(P, E, topk_idx)
    nt = notify(P, E, C, expert_alignment, lay["num_tokens_per_rank"],
                lay["num_tokens_per_expert"], lay["is_token_in_rank"])
    rows = int(nt["part_row_base"][-1])
    dis = dispatch(P, E, H, quant, x_bits, topk_idx, topk_weights, nt["send_head"],
                   nt["part_row_base"], rows)
    return lay, nt, dis
