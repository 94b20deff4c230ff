"""moe_layout_static_scratch: the layout entry point that allocates nothing.

Some callers of the library cannot allocate device memory -- code hosted by an
engine that owns all device memory and forbids allocation after start-up, or
serving loops where cudaMalloc would stall the device. For them the library
keeps the layout's scratch in a buffer compiled into it. These checks call that
entry point through the C ABI and compare it with moe_layout (which takes a
caller-allocated scratch buffer) on two calls in a row with different
routings, so the second call cannot pass on what the first one left behind.
Layout outputs are integers: the comparison is bit-exact.
"""

import ctypes

import numpy as np
import pytest

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


def test_static_scratch_layout_matches_moe_layout_twice():
    import torch

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev).cuda_stream
    cases = [inputs.workload("p128_e256_t512_h7168_zipf", with_x=False, seed=0),
             inputs.workload("p8_e256_t4096_h7168", with_x=False, seed=1)]
    for w in cases:
        shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0)
        # Both shapes' layout partials fit the built-in buffer (the static call
        # below would otherwise return MOE_ERR_UNSUPPORTED); moe_scratch_bytes is
        # larger, as it also covers the other entry points' scratch.
        idx = torch.from_numpy(w.topk_idx).to(dev)
        ref = _outputs(shape, dev)
        scratch = torch.empty(moe.moe_scratch_bytes(shape), dtype=torch.uint8, device=dev)
        moe.moe_layout(shape, idx, ref["num_tokens_per_rank"], ref["num_tokens_per_expert"],
                       ref["is_token_in_rank"], ref["is_token_in_rank_bits"], ref["err"], scratch)
        got = _outputs(shape, dev)
        assert _call_static(shape, idx, got, stream) == moe.MOE_OK
        torch.cuda.synchronize(dev)
        for k in ref:
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(), err_msg=k)
        assert int(got["err"][0].item()) == moe.MOE_OK


def test_static_scratch_rejects_shapes_beyond_its_buffer():
    import torch

    dev = torch.device("cuda", 0)
    # P = 1024 ranks and E = 4096 experts with 64 tokens per rank need ~42 MB of partials.
    shape = moe.make_shape(1024, 4096, 1024 * 64, 8, 64)
    assert moe.moe_scratch_bytes(shape) > moe.MOE_LAYOUT_STATIC_SCRATCH_BYTES
    o = _outputs(shape, dev)   # full-size outputs; the call must leave them untouched
    idx = torch.zeros((shape.S, shape.K), dtype=torch.int32, device=dev)
    st = _call_static(shape, idx, o, torch.cuda.current_stream(dev).cuda_stream)
    assert st == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize(dev)
    assert int(o["err"][0].item()) == -3
