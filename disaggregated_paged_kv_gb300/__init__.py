"""libkvx on GB300: move a finished prefill's KV cache out of a token-paged KV pool.

The C ABI lives in include/kvx.h and libkvx.so (built in-tree by
``disaggregated_paged_kv_gb300.build``); :mod:`disaggregated_paged_kv_gb300.kvx` is its thin
Python binding.
"""
from . import kvx  # noqa: F401
