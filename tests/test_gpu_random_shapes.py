"""Seeded random shapes through every path, against the oracle.

Each shape runs layout -> notify -> dispatch -> combine (rank-major; bf16 or
int8 with the stand-in expert), moe_dispatch_fused where it applies, and the
expert-major path. Every table, every written slot and every combined row is
compared bit for bit (combine also within the 1-ulp bar). The shapes mix
ragged token counts against channel splits, P that are not powers of two,
K up to 16, expert alignment > 1, masked slots, Zipf routing and int8.
"""

import numpy as np
import pytest

from combine_moe_layout_02_gb300 import inputs
from tests import gpu_path as gp
from tests.test_gpu_expert_major import _run as run_expert_major
from tests.test_gpu_fused import _check_fused

pytestmark = pytest.mark.gpu


def _shapes(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 24, 32, 33, 48, 64, 65, 100]))
        E = P * int(rng.integers(1, 9))
        K = int(rng.integers(1, min(16, E) + 1))
        T = int(rng.integers(1, 200))
        quant = int(rng.random() < 0.35)
        H = 16 * int(rng.integers(1, 80)) if quant else 8 * int(rng.integers(1, 160))
        C = int(rng.integers(1, 40))
        A = int(rng.choice([1, 1, 2, 4, 7]))
        mask = float(rng.choice([0.0, 0.0, 0.1, 0.5]))
        routing = "zipf" if rng.random() < 0.3 else "uniform"
        out.append((P, E, T, H, K, quant, C, A, mask, routing, 1000 + i))
    return out


SHAPES = _shapes()


@pytest.mark.parametrize("P,E,T,H,K,quant,C,A,mask,routing,seed", SHAPES,
                         ids=[f"P{s[0]}E{s[1]}T{s[2]}H{s[3]}K{s[4]}q{s[5]}C{s[6]}A{s[7]}" for s in SHAPES])
def test_random_shape_all_paths(P, E, T, H, K, quant, C, A, mask, routing, seed):
    w = inputs.make(P, E, T, H, K, routing=routing, mask_frac=mask, quant=quant, seed=seed, C=C,
                    expert_alignment=A)
    gpu = gp.run_gpu(w, quant=quant, y_mode="int8expert" if quant else "identity")
    assert gpu["layout_err"] == 0 and gpu["dispatch_err"] == 0 and gpu["combine_err"] == 0
    lay, nt = gp.oracle_tables(w)
    gp.assert_tables_equal(gpu, lay, nt)
    gp.compare_dispatch(w, quant, gpu, nt)
    gp.compare_combine(w, gpu, nt)
    if quant == 0 and P <= 64 and E <= 1024 and K <= 16 and P * C <= 4096:
        _check_fused(w)
    run_expert_major(w, quant=quant, y_mode="dequant" if quant else "identity")


def _cluster_shapes(n=12, seed=4049):
    """Longer source ranks (257-2000 tokens): layout in clusters of several
    CTAs and notify's cluster kernel, with its flags kept in registers, kept in
    shared memory or re-read, depending on P and T. Small H keeps the oracle
    quick."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        P = int(rng.choice([2, 6, 8, 12, 24, 33, 48, 64, 65, 100, 128]))
        T = int(rng.integers(257, max(258, min(2000, 40000 // P))))
        E = P * int(rng.integers(1, 5))
        K = int(rng.integers(1, min(16, E) + 1))
        H = 8 * int(rng.integers(1, 33))
        C = int(rng.integers(1, 3 * T // 2))
        A = int(rng.choice([1, 1, 3]))
        mask = float(rng.choice([0.0, 0.1]))
        routing = "zipf" if rng.random() < 0.3 else "uniform"
        out.append((P, E, T, H, K, C, A, mask, routing, 5000 + i))
    return out


CLUSTER_SHAPES = _cluster_shapes()


@pytest.mark.parametrize("P,E,T,H,K,C,A,mask,routing,seed", CLUSTER_SHAPES,
                         ids=[f"P{s[0]}E{s[1]}T{s[2]}H{s[3]}K{s[4]}C{s[5]}A{s[6]}" for s in CLUSTER_SHAPES])
def test_random_long_ranks(P, E, T, H, K, C, A, mask, routing, seed):
    w = inputs.make(P, E, T, H, K, routing=routing, mask_frac=mask, seed=seed, C=C, expert_alignment=A)
    gpu = gp.run_gpu(w)
    assert gpu["layout_err"] == 0 and gpu["dispatch_err"] == 0 and gpu["combine_err"] == 0
    lay, nt = gp.oracle_tables(w)
    gp.assert_tables_equal(gpu, lay, nt)
    gp.compare_dispatch(w, 0, gpu, nt)
    gp.compare_combine(w, gpu, nt)
