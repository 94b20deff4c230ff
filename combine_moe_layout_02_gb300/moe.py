"""ctypes binding of libmoe.so (include/moe.h): argument marshalling only.

Every function here forwards torch tensors' device pointers and the current
CUDA stream to the C ABI of the same name; all work runs in the library's
sm_103a kernels. A non-zero status raises :class:`MoeError`. If the library
has not been built, the first call raises -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_LIBRARY=NAME loads the build variant libmoe_NAME.so (build.py) instead.
LIB_PATH = os.path.join(_HERE, f"libmoe_{os.environ['MOE_LIBRARY']}.so" if os.environ.get("MOE_LIBRARY")
                        else "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_TOPK_OUT_OF_RANGE = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_CUDA = 4
MOE_ERR_UNSUPPORTED = 5
MOE_ERR_DEVICE_TIMEOUT = 6
MOE_ERR_INCONSISTENT = 7

EXPORTS = ("moe_status_string", "moe_check_shape", "moe_slot_stride", "moe_scratch_bytes",
           "moe_max_recv_rows", "moe_layout", "moe_notify", "moe_dispatch", "moe_combine",
           "moe_layout_static_scratch", "moe_pad_partitions", "moe_max_expert_rows",
           "moe_notify_expert", "moe_dispatch_expert", "moe_combine_expert", "moe_dispatch_fused",
           "moe_run_host_workspace_bytes", "moe_run_host", "moe_test_fused_barrier", "moe_exchange_plan")

# moe_run_host flags (include/moe.h).
MOE_RUN_FUSED = 1
MOE_RUN_EXPERT = 2

# Bytes of the scratch buffer built into the library (include/moe.h).
MOE_LAYOUT_STATIC_SCRATCH_BYTES = 1024 * 4


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class moe_shape(ctypes.Structure):
    _fields_ = [("P", ctypes.c_int32), ("E", ctypes.c_int32), ("S", ctypes.c_int32),
                ("K", ctypes.c_int32), ("H", ctypes.c_int32), ("num_channels", ctypes.c_int32),
                ("expert_alignment", ctypes.c_int32), ("quant", ctypes.c_int32)]

    def __repr__(self):
        return "moe_shape(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


def make_shape(P, E, S, K, H, num_channels=16, expert_alignment=1, quant=0) -> moe_shape:
    return moe_shape(P, E, S, K, H, num_channels, expert_alignment, quant)


_lib = None
_lib_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """Open libmoe.so (raises if it is missing)."""
    if _lib is not None:
        return _lib
    with _lib_lock:
        return _lib if _lib is not None else _open_lib()


def _open_lib() -> ctypes.CDLL:
    global _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
    try:  # torch's CUDA runtime satisfies libmoe's libcudart dependency
        import torch  # noqa: F401
    except ImportError:  # pragma: no cover
        pass
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sp = ctypes.POINTER(moe_shape)
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_status_string.argtypes = [i32]
    L.moe_check_shape.restype = i32
    L.moe_check_shape.argtypes = [sp]
    L.moe_slot_stride.restype = i64
    L.moe_slot_stride.argtypes = [i32, i32]
    L.moe_scratch_bytes.restype = i64
    L.moe_scratch_bytes.argtypes = [sp]
    L.moe_max_recv_rows.restype = i64
    L.moe_max_recv_rows.argtypes = [sp]
    L.moe_layout.restype = i32
    L.moe_layout.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, i64, vp]
    L.moe_notify.restype = i32
    L.moe_notify.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp]
    L.moe_dispatch.restype = i32
    L.moe_dispatch.argtypes = [sp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp, vp]
    L.moe_combine.restype = i32
    L.moe_combine.argtypes = [sp, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch_fused.restype = i32
    L.moe_dispatch_fused.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                     vp, i64, vp, vp, vp, vp, vp, i64, vp]
    L.moe_max_expert_rows.restype = i64
    L.moe_max_expert_rows.argtypes = [sp]
    L.moe_notify_expert.restype = i32
    L.moe_notify_expert.argtypes = [sp, vp, vp, vp, vp, vp, vp, i64, vp]
    L.moe_dispatch_expert.restype = i32
    L.moe_dispatch_expert.argtypes = [sp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, vp]
    L.moe_combine_expert.restype = i32
    L.moe_combine_expert.argtypes = [sp, vp, i64, vp, i64, vp, vp, vp, vp, vp, vp]
    L.moe_pad_partitions.restype = i32
    L.moe_pad_partitions.argtypes = [sp, vp, vp, vp, i64, vp, vp, vp, vp]
    L.moe_layout_static_scratch.restype = i32
    L.moe_layout_static_scratch.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_run_host_workspace_bytes.restype = i64
    L.moe_run_host_workspace_bytes.argtypes = [sp, i32]
    L.moe_run_host.restype = i32
    L.moe_run_host.argtypes = [sp, i32, vp, vp, vp, vp, vp, i64, i32, vp, i64, vp]
    L.moe_test_fused_barrier.restype = i32
    L.moe_test_fused_barrier.argtypes = [ctypes.c_uint32, i32]
    L.moe_exchange_plan.restype = i32
    L.moe_exchange_plan.argtypes = [sp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _ptr(t):
    """Device pointer of a tensor (None -> NULL). Accepts raw ints too."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def moe_check_shape(shape: moe_shape) -> int:
    return int(lib().moe_check_shape(ctypes.byref(shape)))


def moe_slot_stride(H: int, quant: int) -> int:
    return int(lib().moe_slot_stride(int(H), int(quant)))


def moe_scratch_bytes(shape: moe_shape) -> int:
    return int(lib().moe_scratch_bytes(ctypes.byref(shape)))


def moe_max_recv_rows(shape: moe_shape) -> int:
    return int(lib().moe_max_recv_rows(ctypes.byref(shape)))


def moe_layout(shape, topk_idx, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
               is_token_in_rank_bits, err, scratch, stream=None):
    st = lib().moe_layout(ctypes.byref(shape), _ptr(topk_idx), _ptr(num_tokens_per_rank),
                          _ptr(num_tokens_per_expert), _ptr(is_token_in_rank),
                          _ptr(is_token_in_rank_bits), _ptr(err), _ptr(scratch),
                          int(scratch.numel() * scratch.element_size()), _stream(stream))
    _check(st, "moe_layout")


def moe_notify(shape, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
               rank_prefix_matrix, channel_prefix_matrix, recv_channel_prefix_matrix,
               num_recv_tokens, num_recv_tokens_per_expert, recv_expert_offset, send_head,
               part_row_base, scratch, stream=None):
    st = lib().moe_notify(ctypes.byref(shape), _ptr(num_tokens_per_rank), _ptr(num_tokens_per_expert),
                          _ptr(is_token_in_rank), _ptr(rank_prefix_matrix),
                          _ptr(channel_prefix_matrix), _ptr(recv_channel_prefix_matrix),
                          _ptr(num_recv_tokens), _ptr(num_recv_tokens_per_expert),
                          _ptr(recv_expert_offset), _ptr(send_head), _ptr(part_row_base),
                          _ptr(scratch), int(scratch.numel() * scratch.element_size()),
                          _stream(stream))
    _check(st, "moe_notify")


def moe_dispatch(shape, x, topk_idx, topk_weights, send_head, part_row_base, recv_arena, arena_rows,
                 recv_src_idx, recv_topk_idx, recv_topk_weights, err, stream=None):
    st = lib().moe_dispatch(ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(topk_weights),
                            _ptr(send_head), _ptr(part_row_base), _ptr(recv_arena), int(arena_rows),
                            _ptr(recv_src_idx), _ptr(recv_topk_idx), _ptr(recv_topk_weights),
                            _ptr(err), _stream(stream))
    _check(st, "moe_dispatch")


def moe_combine(shape, y, y_row_stride, part_row_base, arena_rows, send_head, topk_idx,
                topk_weights, out, err, stream=None):
    st = lib().moe_combine(ctypes.byref(shape), _ptr(y), int(y_row_stride), _ptr(part_row_base),
                           int(arena_rows), _ptr(send_head), _ptr(topk_idx), _ptr(topk_weights),
                           _ptr(out), _ptr(err), _stream(stream))
    _check(st, "moe_combine")


def moe_dispatch_fused(shape, x, topk_idx, topk_weights, num_tokens_per_rank, num_tokens_per_expert,
                       is_token_in_rank, is_token_in_rank_bits, rank_prefix_matrix, channel_prefix_matrix,
                       recv_channel_prefix_matrix, num_recv_tokens, num_recv_tokens_per_expert,
                       recv_expert_offset, send_head, part_row_base, recv_arena, arena_rows, recv_src_idx,
                       recv_topk_idx, recv_topk_weights, err, scratch, stream=None):
    st = lib().moe_dispatch_fused(
        ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(topk_weights), _ptr(num_tokens_per_rank),
        _ptr(num_tokens_per_expert), _ptr(is_token_in_rank), _ptr(is_token_in_rank_bits),
        _ptr(rank_prefix_matrix), _ptr(channel_prefix_matrix), _ptr(recv_channel_prefix_matrix),
        _ptr(num_recv_tokens), _ptr(num_recv_tokens_per_expert), _ptr(recv_expert_offset), _ptr(send_head),
        _ptr(part_row_base), _ptr(recv_arena), int(arena_rows), _ptr(recv_src_idx), _ptr(recv_topk_idx),
        _ptr(recv_topk_weights), _ptr(err), _ptr(scratch), int(scratch.numel() * scratch.element_size()),
        _stream(stream))
    _check(st, "moe_dispatch_fused")


def moe_max_expert_rows(shape: moe_shape) -> int:
    return int(lib().moe_max_expert_rows(ctypes.byref(shape)))


def moe_notify_expert(shape, topk_idx, num_recv_tokens_per_expert, recv_expert_offset, slot_row,
                      expert_part_base, scratch, stream=None):
    st = lib().moe_notify_expert(ctypes.byref(shape), _ptr(topk_idx), _ptr(num_recv_tokens_per_expert),
                                 _ptr(recv_expert_offset), _ptr(slot_row), _ptr(expert_part_base),
                                 _ptr(scratch), int(scratch.numel() * scratch.element_size()),
                                 _stream(stream))
    _check(st, "moe_notify_expert")


def moe_dispatch_expert(shape, x, topk_idx, topk_weights, slot_row, expert_part_base, recv_arena,
                        arena_rows, recv_src_idx, recv_weight, err, stream=None):
    st = lib().moe_dispatch_expert(ctypes.byref(shape), _ptr(x), _ptr(topk_idx), _ptr(topk_weights),
                                   _ptr(slot_row), _ptr(expert_part_base), _ptr(recv_arena),
                                   int(arena_rows), _ptr(recv_src_idx), _ptr(recv_weight), _ptr(err),
                                   _stream(stream))
    _check(st, "moe_dispatch_expert")


def moe_combine_expert(shape, y, y_row_stride, expert_part_base, arena_rows, slot_row, topk_idx,
                       topk_weights, out, err, stream=None):
    st = lib().moe_combine_expert(ctypes.byref(shape), _ptr(y), int(y_row_stride),
                                  _ptr(expert_part_base), int(arena_rows), _ptr(slot_row),
                                  _ptr(topk_idx), _ptr(topk_weights), _ptr(out), _ptr(err),
                                  _stream(stream))
    _check(st, "moe_combine_expert")


def moe_pad_partitions(shape, num_recv_tokens, part_row_base, recv_arena, arena_rows,
                       recv_src_idx, recv_topk_idx, recv_topk_weights, stream=None):
    st = lib().moe_pad_partitions(ctypes.byref(shape), _ptr(num_recv_tokens), _ptr(part_row_base),
                                  _ptr(recv_arena), int(arena_rows), _ptr(recv_src_idx),
                                  _ptr(recv_topk_idx), _ptr(recv_topk_weights), _stream(stream))
    _check(st, "moe_pad_partitions")


def moe_layout_static_scratch(shape, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                              is_token_in_rank, is_token_in_rank_bits, err, stream=None):
    """moe_layout using the library's built-in scratch buffer: for callers that
    cannot allocate device memory (see include/moe.h). Calls must not overlap
    on the GPU; the first call on a device must precede any stream capture."""
    st = lib().moe_layout_static_scratch(ctypes.byref(shape), _ptr(topk_idx), _ptr(num_tokens_per_rank),
                                         _ptr(num_tokens_per_expert), _ptr(is_token_in_rank),
                                         _ptr(is_token_in_rank_bits), _ptr(err), _stream(stream))
    _check(st, "moe_layout_static_scratch")


def _host_ptr(t):
    """Host address of a contiguous CPU tensor or numpy array (None -> NULL)."""
    if t is None:
        return None
    if hasattr(t, "is_cuda"):
        if t.is_cuda:
            raise ValueError("expected a host tensor")
        if not t.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        return t.data_ptr()
    if not t.flags["C_CONTIGUOUS"]:
        raise ValueError("expected a contiguous array")
    return t.ctypes.data


def moe_test_fused_barrier(spin_limit: int, skip_cta: int) -> None:
    """Arm the next moe_dispatch_fused call of this thread with a short grid
    barrier and (skip_cta >= 0) one CTA that leaves out its first arrival, so
    that its bounded waits run out (a test of the timeout path)."""
    _check(lib().moe_test_fused_barrier(int(spin_limit), int(skip_cta)), "moe_test_fused_barrier")


def moe_exchange_plan(shape: moe_shape, self_rank: int, ntpr_all, ntpe_all) -> dict:
    """What rank self_rank needs from every rank's gathered layout rows (host
    numpy arrays ntpr_all [P,P], ntpe_all [P,E]); the C function computes it on
    the host (include/moe.h)."""
    import numpy as np

    P, E = shape.P, shape.E
    ntpr = np.ascontiguousarray(ntpr_all, np.int32)
    ntpe = np.ascontiguousarray(ntpe_all, np.int32)
    if ntpr.shape != (P, P) or ntpe.shape != (P, E):
        raise ValueError("expected ntpr_all [P,P] and ntpe_all [P,E]")
    out = dict(rank_prefix_matrix=np.empty((P, P), np.int32), num_recv_tokens=np.empty((P,), np.int32),
               send_row_base=np.empty((P,), np.int64),
               num_recv_tokens_per_expert=np.empty((E // P,), np.int32),
               recv_expert_offset=np.empty((E // P,), np.int32), part_row_base=np.empty((P + 1,), np.int64))
    h = lambda a: a.ctypes.data
    _check(lib().moe_exchange_plan(ctypes.byref(shape), int(self_rank), h(ntpr), h(ntpe),
                                   h(out["rank_prefix_matrix"]), h(out["num_recv_tokens"]), h(out["send_row_base"]),
                                   h(out["num_recv_tokens_per_expert"]), h(out["recv_expert_offset"]),
                                   h(out["part_row_base"])), "moe_exchange_plan")
    return out


def exchange_counts(shape: moe_shape, num_tokens_per_rank_row, num_tokens_per_expert_row, group=None) -> dict:
    """The count exchange of a path spread over the ranks of a torch.distributed
    group (one expert-parallel rank per process, group size = shape.P): this
    rank's rows of num_tokens_per_rank [P] and num_tokens_per_expert [E] (from
    moe_layout over its own tokens) are all-gathered in rank order, then
    moe_exchange_plan gives this rank's plan. The gathered tables are returned
    too (ntpr_all, ntpe_all)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if world != shape.P:
        raise ValueError(f"group of {world} ranks for P = {shape.P}")
    row = torch.cat([torch.as_tensor(num_tokens_per_rank_row).reshape(-1).to(torch.int32),
                     torch.as_tensor(num_tokens_per_expert_row).reshape(-1).to(torch.int32)])
    if row.numel() != shape.P + shape.E:
        raise ValueError("expected rows of P and E counts")
    parts = [torch.empty_like(row) for _ in range(world)]
    dist.all_gather(parts, row.contiguous(), group=group)
    table = torch.stack(parts).cpu().numpy()
    ntpr_all, ntpe_all = table[:, :shape.P], table[:, shape.P:]
    plan = moe_exchange_plan(shape, rank, ntpr_all, ntpe_all)
    plan.update(ntpr_all=ntpr_all, ntpe_all=ntpe_all)
    return plan


def moe_run_host_workspace_bytes(shape: moe_shape, n_batches: int) -> int:
    return int(lib().moe_run_host_workspace_bytes(ctypes.byref(shape), int(n_batches)))


def moe_run_host(shape: moe_shape, x_host, topk_idx_host, topk_weights_host, out_host, workspace,
                 y=None, y_row_stride=0, fused=False, expert=False, err_host=None):
    """Run the path over len(x_host) host-resident batches end to end.

    x_host / topk_idx_host / out_host: sequences of host tensors (pinned for
    overlap), one per batch; topk_weights_host: such a sequence or None.
    workspace: device uint8 tensor of moe_run_host_workspace_bytes bytes.
    err_host: None or an int32 numpy array of n batches (device error words).
    Blocking; raises MoeError on any non-OK status.
    """
    n = len(x_host)
    if len(topk_idx_host) != n or len(out_host) != n or (topk_weights_host is not None
                                                         and len(topk_weights_host) != n):
        raise ValueError("one entry per batch in every host list")
    arr = ctypes.c_void_p * max(n, 1)
    xs = arr(*[_host_ptr(t) for t in x_host])
    ids = arr(*[_host_ptr(t) for t in topk_idx_host])
    ws = arr(*[_host_ptr(t) for t in topk_weights_host]) if topk_weights_host is not None else None
    outs = arr(*[_host_ptr(t) for t in out_host])
    eh = None
    if err_host is not None:
        if err_host.dtype.itemsize != 4 or err_host.size < n:
            raise ValueError("err_host: int32 array of one entry per batch")
        eh = err_host.ctypes.data
    st = lib().moe_run_host(ctypes.byref(shape), n, ctypes.cast(xs, ctypes.c_void_p),
                            ctypes.cast(ids, ctypes.c_void_p),
                            ctypes.cast(ws, ctypes.c_void_p) if ws is not None else None,
                            ctypes.cast(outs, ctypes.c_void_p), _ptr(y), int(y_row_stride),
                            (MOE_RUN_FUSED if fused else 0) | (MOE_RUN_EXPERT if expert else 0), _ptr(workspace),
                            workspace.numel(), eh)
    _check(st, "moe_run_host")


class Buffers:
    """Device buffers for one shape, allocated with torch (memory only).

    ``arena_rows`` defaults to :func:`moe_max_recv_rows`, which always holds
    the packed partitions moe_notify lays out, so no host read-back of the
    receive counts is needed before dispatch.
    """

    def __init__(self, shape: moe_shape, device="cuda", arena_rows: int | None = None,
                 side_arrays: bool = True, bits: bool = True):
        import torch

        P, E, S, K, H, C = shape.P, shape.E, shape.S, shape.K, shape.H, shape.num_channels
        self.shape = shape
        self.device = device
        i32, dev = torch.int32, device
        self.num_tokens_per_rank = torch.empty((P, P), dtype=i32, device=dev)
        self.num_tokens_per_expert = torch.empty((P, E), dtype=i32, device=dev)
        self.is_token_in_rank = torch.empty((S, P), dtype=torch.uint8, device=dev)
        self.is_token_in_rank_bits = (torch.empty((S, (P + 31) // 32), dtype=i32, device=dev)
                                      if bits else None)
        self.err = torch.zeros((4,), dtype=i32, device=dev)
        self.scratch = torch.empty((max(moe_scratch_bytes(shape), 256),), dtype=torch.uint8, device=dev)
        self.rank_prefix_matrix = torch.empty((P, P), dtype=i32, device=dev)
        self.channel_prefix_matrix = torch.empty((P, P, C), dtype=i32, device=dev)
        self.recv_channel_prefix_matrix = torch.empty((P, P, C), dtype=i32, device=dev)
        self.num_recv_tokens = torch.empty((P,), dtype=i32, device=dev)
        self.num_recv_tokens_per_expert = torch.empty((P, E // P), dtype=i32, device=dev)
        self.recv_expert_offset = torch.empty((P, E // P), dtype=i32, device=dev)
        self.send_head = torch.empty((S, P), dtype=i32, device=dev)
        self.part_row_base = torch.empty((P + 1,), dtype=torch.int64, device=dev)
        self.arena_rows = moe_max_recv_rows(shape) if arena_rows is None else int(arena_rows)
        self.stride = moe_slot_stride(H, shape.quant)
        self.recv_arena = torch.empty((max(self.arena_rows, 1), self.stride), dtype=torch.uint8, device=dev)
        if side_arrays:
            self.recv_src_idx = torch.empty((max(self.arena_rows, 1),), dtype=i32, device=dev)
            self.recv_topk_idx = torch.empty((max(self.arena_rows, 1), K), dtype=i32, device=dev)
            self.recv_topk_weights = torch.empty((max(self.arena_rows, 1), K), dtype=torch.float32,
                                                 device=dev)
        else:
            self.recv_src_idx = self.recv_topk_idx = self.recv_topk_weights = None

    def layout(self, topk_idx, stream=None):
        moe_layout(self.shape, topk_idx, self.num_tokens_per_rank, self.num_tokens_per_expert,
                   self.is_token_in_rank, self.is_token_in_rank_bits, self.err, self.scratch, stream)

    def notify(self, stream=None):
        moe_notify(self.shape, self.num_tokens_per_rank, self.num_tokens_per_expert,
                   self.is_token_in_rank, self.rank_prefix_matrix, self.channel_prefix_matrix,
                   self.recv_channel_prefix_matrix, self.num_recv_tokens,
                   self.num_recv_tokens_per_expert, self.recv_expert_offset, self.send_head,
                   self.part_row_base, self.scratch, stream)

    def dispatch(self, x, topk_idx, topk_weights, stream=None):
        moe_dispatch(self.shape, x, topk_idx, topk_weights, self.send_head, self.part_row_base,
                     self.recv_arena, self.arena_rows, self.recv_src_idx, self.recv_topk_idx,
                     self.recv_topk_weights, self.err, stream)

    def combine(self, out, topk_idx, topk_weights, y=None, y_row_stride=None, stream=None):
        """Combine; by default y is the dispatch arena (identity experts)."""
        if y is None:
            y, y_row_stride = self.recv_arena, self.stride
        moe_combine(self.shape, y, y_row_stride, self.part_row_base, self.arena_rows, self.send_head,
                    topk_idx, topk_weights, out, self.err, stream)

    def pad(self, stream=None):
        """Pad fixed-capacity partitions past their received counts."""
        moe_pad_partitions(self.shape, self.num_recv_tokens, self.part_row_base, self.recv_arena,
                           self.arena_rows, self.recv_src_idx, self.recv_topk_idx,
                           self.recv_topk_weights, stream)

    # ---- expert-major layout (after layout and notify) --------------------
    def _expert_buffers(self, arena_rows=None):
        import torch

        if getattr(self, "slot_row", None) is not None:
            return
        s, dev = self.shape, self.device
        self.slot_row = torch.empty((s.S, s.K), dtype=torch.int32, device=dev)
        self.expert_part_base = torch.empty((s.P + 1,), dtype=torch.int64, device=dev)
        self.expert_rows = moe_max_expert_rows(s) if arena_rows is None else int(arena_rows)
        rows = max(self.expert_rows, 1)
        self.expert_arena = torch.empty((rows, self.stride), dtype=torch.uint8, device=dev)
        self.expert_src_idx = torch.empty((rows,), dtype=torch.int32, device=dev)
        self.expert_weight = torch.empty((rows,), dtype=torch.float32, device=dev)

    def notify_expert(self, topk_idx, stream=None, arena_rows=None):
        self._expert_buffers(arena_rows)
        moe_notify_expert(self.shape, topk_idx, self.num_recv_tokens_per_expert, self.recv_expert_offset,
                          self.slot_row, self.expert_part_base, self.scratch, stream)

    def dispatch_expert(self, x, topk_idx, topk_weights, stream=None):
        moe_dispatch_expert(self.shape, x, topk_idx, topk_weights, self.slot_row, self.expert_part_base,
                            self.expert_arena, self.expert_rows, self.expert_src_idx, self.expert_weight,
                            self.err, stream)

    def combine_expert(self, out, topk_idx, topk_weights, y=None, y_row_stride=None, stream=None):
        """Per-slot combine; by default y is the expert-major arena (identity experts)."""
        if y is None:
            y, y_row_stride = self.expert_arena, self.stride
        moe_combine_expert(self.shape, y, y_row_stride, self.expert_part_base, self.expert_rows,
                           self.slot_row, topk_idx, topk_weights, out, self.err, stream)

    def dispatch_fused(self, x, topk_idx, topk_weights, stream=None):
        """layout + notify + dispatch in one launch (small shapes only)."""
        moe_dispatch_fused(self.shape, x, topk_idx, topk_weights, self.num_tokens_per_rank,
                           self.num_tokens_per_expert, self.is_token_in_rank, self.is_token_in_rank_bits,
                           self.rank_prefix_matrix, self.channel_prefix_matrix,
                           self.recv_channel_prefix_matrix, self.num_recv_tokens,
                           self.num_recv_tokens_per_expert, self.recv_expert_offset, self.send_head,
                           self.part_row_base, self.recv_arena, self.arena_rows, self.recv_src_idx,
                           self.recv_topk_idx, self.recv_topk_weights, self.err, self.scratch, stream)

    def step(self, x, topk_idx, topk_weights, out, stream=None):
        """One pass of the hot path: layout -> notify -> dispatch -> combine."""
        self.layout(topk_idx, stream)
        self.notify(stream)
        self.dispatch(x, topk_idx, topk_weights, stream)
        self.combine(out, topk_idx, topk_weights, stream=stream)
