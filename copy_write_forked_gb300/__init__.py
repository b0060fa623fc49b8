"""GB300-native copy-on-write tree KV cache with tree-aware decode attention.

The compute path lives in the C-ABI library ``libdendrite.so`` (hand-written
CUDA for sm_103a, built in-tree); :mod:`.dendrite` is its thin ctypes binding.
"""
from .dendrite import Pool, DendriteError, lib, plan_segments  # noqa: F401

__version__ = "0.1.0"
