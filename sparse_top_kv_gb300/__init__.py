"""sparse_top_kv_gb300 -- GB300-native (sm_103a) HiSparse top-k sparse decode.

The hot path lives in libhs.so (C ABI: include/hs_api.h); `hs` is its thin
Python binding, `pipeline` strings the four stages into one decode step, and
`inputs` holds the seeded synthetic workload generators.
"""
from . import hs  # noqa: F401

__all__ = ["hs"]
