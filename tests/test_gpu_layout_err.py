"""moe_layout's error word under CUDA graph replay and for both kinds of
source rank: held by one CTA (no cluster exchange) or by a thread-block
cluster. Each source rank writes an out-of-range flag to scratch and a
one-block kernel folds the flags into err.

moe_layout is captured once in a CUDA graph and replayed with the routing
changed in place between replays (clean, one bad id, clean, a bad id on every
source rank twice, clean), so a replay passes only if it writes err from its
own flags. The last replay's tables are compared with the oracle. Integers:
exact.
"""

import numpy as np
import pytest

import oracle
from combine_moe_layout_02_gb300 import inputs, moe

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["p32_e256_t128_h1024", "p8_e256_t4096_h7168", "tiny_p4_e16_h256"])
def test_error_word_across_graph_replays(name):
    import torch

    dev = torch.device("cuda", 0)
    w = inputs.workload(name, with_x=False, seed=3)
    shape = moe.make_shape(w.P, w.E, w.S, w.K, w.H, w.C, w.expert_alignment, 0)
    buf = moe.Buffers(shape, dev)
    idx = torch.from_numpy(w.topk_idx).to(dev)
    clean = idx.clone()
    one_bad = clean.clone()
    one_bad[w.S // 2, 0] = w.E
    all_bad = clean.clone()
    T = w.S // w.P
    all_bad[torch.arange(w.P, device=dev) * T, w.K - 1] = w.E + 7

    buf.err.fill_(-5)
    buf.layout(idx)  # outside the graph first (kernels loaded and configured)
    torch.cuda.synchronize(dev)
    assert int(buf.err[0].item()) == moe.MOE_OK
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        buf.layout(idx, torch.cuda.current_stream(dev))
    torch.cuda.current_stream(dev).wait_stream(cap)
    expect = []
    for src, code in ((clean, moe.MOE_OK), (one_bad, moe.MOE_ERR_TOPK_OUT_OF_RANGE), (clean, moe.MOE_OK),
                      (all_bad, moe.MOE_ERR_TOPK_OUT_OF_RANGE), (all_bad, moe.MOE_ERR_TOPK_OUT_OF_RANGE),
                      (clean, moe.MOE_OK)):
        idx.copy_(src)
        buf.err.fill_(-5)
        graph.replay()
        torch.cuda.synchronize(dev)
        expect.append((int(buf.err[0].item()), code))
    assert [g for g, _ in expect] == [c for _, c in expect]
    lay = oracle.layout(w.P, w.E, w.topk_idx)
    for k in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank"):
        np.testing.assert_array_equal(getattr(buf, k).cpu().numpy(), lay[k], err_msg=k)
