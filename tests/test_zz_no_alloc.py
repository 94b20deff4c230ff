"""moe_layout_static_scratch: the layout entry point that allocates nothing.

Some callers of the library cannot allocate device memory -- code hosted by an
engine that owns all device memory and forbids allocation after start-up, or
serving loops where cudaMalloc would stall the device. For them the library
keeps the layout's scratch (one out-of-range flag per source rank) in a buffer
compiled into it. These checks call that entry point through the C ABI and
compare it with moe_layout (which takes a caller-allocated scratch buffer) and
with the oracle, on calls in a row with different routings, so no call can
pass on what an earlier one left behind in the shared buffer. Layout outputs
are integers: the comparison is bit-exact.
"""

import ctypes

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs, moe

pytestmark = pytest.mark.gpu


def _outputs(shape, dev):
    import torch

    P, E, S = shape.P, shape.E, shape.S
    return dict(
        num_tokens_per_rank=torch.full((P, P), -3, dtype=torch.int32, device=dev),
        num_tokens_per_expert=torch.full((P, E), -3, dtype=torch.int32, device=dev),
        is_token_in_rank=torch.full((S, P), 7, dtype=torch.uint8, device=dev),
        is_token_in_rank_bits=torch.full((S, (P + 31) // 32), -3, dtype=torch.int32, device=dev),
        err=torch.full((1,), -3, dtype=torch.int32, device=dev),
    )


def _call_static(shape, idx, o, stream):
    """Straight through the C ABI, no Python helper in between."""
    return moe.lib().moe_layout_static_scratch(
        ctypes.byref(shape), ctypes.c_void_p(idx.data_ptr()),
        ctypes.c_void_p(o["num_tokens_per_rank"].data_ptr()),
        ctypes.c_void_p(o["num_tokens_per_expert"].data_ptr()),
        ctypes.c_void_p(o["is_token_in_rank"].data_ptr()),
        ctypes.c_void_p(o["is_token_in_rank_bits"].data_ptr()),
        ctypes.c_void_p(o["err"].data_ptr()), ctypes.c_void_p(stream))


def _check_against_oracle(w, got):
    lay = oracle.layout(w.P, w.E, w.topk_idx)
    for k in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank"):
        np.testing.assert_array_equal(got[k].cpu().numpy(), lay[k], err_msg=k)
    bits = np.zeros((w.S, (w.P + 31) // 32), dtype=np.uint32)
    for d in range(w.P):
        bits[:, d // 32] |= lay["is_token_in_rank"][:, d].astype(np.uint32) << np.uint32(d % 32)
    np.testing.assert_array_equal(got["is_token_in_rank_bits"].cpu().numpy().view(np.uint32), bits)


def test_static_scratch_layout_matches_moe_layout_and_oracle():
    import torch

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev).cuda_stream
    # Three static calls in a row on one stream. The second has another shape;
    # the third repeats the first shape with another routing and is enqueued
    # directly behind the second, with no synchronisation in between.
    ws = [inputs.workload("p128_e256_t512_h7168_zipf", with_x=False, seed=0),
          inputs.workload("p8_e256_t4096_h7168", with_x=False, seed=1),
          inputs.workload("p128_e256_t512_h7168_zipf", with_x=False, seed=5)]
    shapes = [moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0) for w in ws]
    idxs = [torch.from_numpy(w.topk_idx).to(dev) for w in ws]
    refs = []
    for w, shape, idx in zip(ws, shapes, idxs):
        ref = _outputs(shape, dev)
        scratch = torch.empty(moe.moe_scratch_bytes(shape), dtype=torch.uint8, device=dev)
        moe.moe_layout(shape, idx, ref["num_tokens_per_rank"], ref["num_tokens_per_expert"],
                       ref["is_token_in_rank"], ref["is_token_in_rank_bits"], ref["err"], scratch)
        refs.append(ref)
    torch.cuda.synchronize(dev)
    gots = [_outputs(shape, dev) for shape in shapes]
    assert _call_static(shapes[0], idxs[0], gots[0], stream) == moe.MOE_OK
    torch.cuda.synchronize(dev)
    assert _call_static(shapes[1], idxs[1], gots[1], stream) == moe.MOE_OK
    assert _call_static(shapes[2], idxs[2], gots[2], stream) == moe.MOE_OK
    torch.cuda.synchronize(dev)
    for w, ref, got in zip(ws, refs, gots):
        for k in ref:
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(), err_msg=k)
        assert int(got["err"][0].item()) == moe.MOE_OK
        _check_against_oracle(w, got)


def test_static_scratch_reports_out_of_range_ids():
    """The flags in the shared buffer carry an out-of-range id into err, and the
    next clean call on the same stream clears it again; a bad id on several
    source ranks at once, and on the last one alone, is reported as well."""
    import torch

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev).cuda_stream
    w = inputs.workload("p32_e256_t128_h1024", with_x=False, seed=2)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0)
    bad = w.topk_idx.copy()
    bad[17, 3] = w.E  # one id past the last expert, on source rank 0
    many = w.topk_idx.copy()
    T = w.S // w.P
    for s_ in (0, 5, w.P - 1):
        many[s_ * T + 3, 0] = w.E + s_
    last = w.topk_idx.copy()
    last[w.S - 1, w.K - 1] = 1 << 30  # the last source rank alone
    o_bad, o_ok, o_many, o_last, o_ok2 = (_outputs(shape, dev) for _ in range(5))
    for arr, o in ((bad, o_bad), (w.topk_idx, o_ok), (many, o_many), (last, o_last), (w.topk_idx, o_ok2)):
        assert _call_static(shape, torch.from_numpy(arr).to(dev), o, stream) == moe.MOE_OK
    torch.cuda.synchronize(dev)
    assert int(o_bad["err"][0].item()) == moe.MOE_ERR_TOPK_OUT_OF_RANGE
    assert int(o_ok["err"][0].item()) == moe.MOE_OK
    assert int(o_many["err"][0].item()) == moe.MOE_ERR_TOPK_OUT_OF_RANGE
    assert int(o_last["err"][0].item()) == moe.MOE_ERR_TOPK_OUT_OF_RANGE
    assert int(o_ok2["err"][0].item()) == moe.MOE_OK
    _check_against_oracle(w, o_ok)
    _check_against_oracle(w, o_ok2)


def test_static_scratch_rejects_shapes_beyond_its_buffer():
    import torch

    dev = torch.device("cuda", 0)
    # P = 2048 source ranks would need 8 KB of flags, past the 4 KB buffer
    # (and past MOE_MAX_RANKS): refused before anything is enqueued.
    shape = moe.make_shape(2048, 4096, 2048 * 4, 8, 64)
    o = _outputs(moe.make_shape(4, 16, 64, 8, 64), dev)  # never written
    idx = torch.zeros((shape.S, shape.K), dtype=torch.int32, device=dev)
    st = _call_static(shape, idx, o, torch.cuda.current_stream(dev).cuda_stream)
    assert st == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize(dev)
    assert int(o["err"][0].item()) == -3
