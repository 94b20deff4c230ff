"""Small numpy/torch helpers shared by the tests (no path arithmetic here)."""

from __future__ import annotations

import numpy as np


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to binary32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits_torch(values: np.ndarray) -> np.ndarray:
    """bfloat16 round-to-nearest-even through torch's own conversion."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(values, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between two bfloat16 arrays.

    Bit patterns are mapped to a monotone integer line (sign-magnitude to
    two's complement), so +0 and -0 are one apart and neighbours are one apart.
    """
    def key(x):
        x = np.asarray(x, np.uint16).astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF) - 1, x)

    return np.abs(key(a_bits) - key(b_bits))


def channel_sizes(T: int, C: int) -> list[int]:
    """Sizes of numpy's array_split of T items into C parts (larger parts first)."""
    return [len(a) for a in np.array_split(np.arange(T), C)]


def stable_receive_rows(itr: np.ndarray) -> np.ndarray:
    """Row of each (g, d) in d's partition when pairs are stably sorted by d.

    Returns an int32 [S, P] array with -1 where itr is 0. Built from
    numpy's stable argsort, independently of any running counter.
    """
    S, P = itr.shape
    g_idx, d_idx = np.nonzero(itr)
    order = np.argsort(d_idx, kind="stable")
    d_sorted = d_idx[order]
    g_sorted = g_idx[order]
    starts = np.searchsorted(d_sorted, np.arange(P), side="left")
    pos = np.arange(d_sorted.shape[0]) - starts[d_sorted]
    out = np.full((S, P), -1, np.int32)
    out[g_sorted, d_sorted] = pos
    return out
