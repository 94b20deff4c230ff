"""Concurrent callers: host threads, each with its own CUDA stream and buffers.

The library keeps one process-wide launch cache: each kernel's shared-memory
allowance and occupancy, per device. Here several threads run the path at
the same time, each on its own stream. Their shapes need different
shared-memory sizes for the same kernels, so the cache is read and grown
under contention while the other threads' launches are in flight. ctypes
releases the GIL around every call, so the C entry points really do run
concurrently.

Every thread's tables, dispatched rows and combined outputs must equal the
oracle's bit for bit, and every error word must stay clear.
"""

import threading

import numpy as np
import pytest

from combine_moe_layout_02_gb300 import inputs, moe
from tests import gpu_path as gp

pytestmark = pytest.mark.gpu

# (P, E, T, H, K, quant). The dispatch ring depth and the combine kernel
# instantiation differ between these.
CASES = [
    (8, 64, 96, 7168, 8, 0),
    (4, 16, 64, 256, 2, 0),
    (16, 128, 40, 2048, 6, 1),
    (32, 256, 24, 4096, 8, 0),
]
REPEATS = 12


def _worker(i, case, start, results):
    import torch

    P, E, T, H, K, quant = case
    try:
        dev = torch.device("cuda", 0)
        w = inputs.make(P, E, T, H, K, seed=70 + i, quant=quant, mask_frac=0.05)
        shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, quant)
        st = torch.cuda.Stream(dev)
        with torch.cuda.stream(st):
            buf = moe.Buffers(shape, dev)
            x = torch.from_numpy(w.x_bits.view(np.int16)).to(dev)
            idx = torch.from_numpy(np.ascontiguousarray(w.topk_idx, np.int32)).to(dev)
            wts = torch.from_numpy(w.topk_weights).to(dev)
            out = torch.empty((w.S, w.H), dtype=torch.int16, device=dev)
            if quant:
                # int8 slots: combine reads bf16 expert outputs, here fresh rows
                g = torch.Generator(device="cpu").manual_seed(500 + i)
                y = torch.randn((max(buf.arena_rows, 1), w.H), generator=g).to(torch.bfloat16)
                y = y.view(torch.int16).to(dev)
                y_stride = 2 * w.H
            else:
                y, y_stride = buf.recv_arena, buf.stride
        st.synchronize()
        start.wait()
        for _ in range(REPEATS):
            buf.layout(idx, st)
            buf.notify(st)
            buf.dispatch(x, idx, wts, st)
            moe.moe_combine(shape, y, y_stride, buf.part_row_base, buf.arena_rows, buf.send_head, idx, wts,
                            out, buf.err, st)
        st.synchronize()
        res = {k: getattr(buf, k).cpu().numpy() for k in gp.LAYOUT_KEYS + gp.NOTIFY_KEYS}
        res["is_token_in_rank_bits"] = res["is_token_in_rank_bits"].view(np.uint32)
        res.update(out=out.cpu().numpy().view(np.uint16), err=buf.err.cpu().numpy(), buf=buf, y=y,
                   y_stride=y_stride, w=w)
        results[i] = res
    except BaseException as e:  # reported by the main thread
        results[i] = e


def test_threads_on_separate_streams_match_the_oracle():
    results = [None] * len(CASES)
    start = threading.Barrier(len(CASES))
    threads = [threading.Thread(target=_worker, args=(i, c, start, results)) for i, c in enumerate(CASES)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
        assert not t.is_alive(), "a worker thread did not finish"
    for (P, E, T, H, K, quant), res in zip(CASES, results):
        if isinstance(res, BaseException):
            raise res
        w = res["w"]
        assert not res["err"].any(), f"device error word set: {res['err']}"
        lay, nt = gp.oracle_tables(w)
        gp.assert_tables_equal(res, lay, nt)
        dis_err, _ = gp.compare_dispatch(w, quant, res, nt)
        assert dis_err == 0
        gp.compare_combine(w, res, nt)
