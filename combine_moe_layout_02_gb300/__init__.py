"""GB300-native MoE dispatch/combine hot path.

The compute path is the C-ABI library ``libmoe.so`` built from ``csrc/``
(hand-written CUDA for sm_103a). ``moe`` is its thin ctypes binding;
``inputs`` draws the seeded synthetic workloads. Importing the package loads
nothing; the library is opened on first use and a missing library raises.
"""

__all__ = ["moe", "inputs"]
