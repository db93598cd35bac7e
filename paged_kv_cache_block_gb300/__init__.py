"""GB300-native paged KV cache decode path.

``paged_kv_cache_block_gb300.kvcache`` is the Python binding of the C-ABI library
``libpagedkv.so`` (slot mapping, cache write, paged decode attention); importing it loads the
library and fails loudly if it has not been built.  ``paged_kv_cache_block_gb300.workloads``
holds the seeded synthetic decode batches.
"""
__version__ = "0.1.0"
