"""Paged decode attention for GB300 (sm_103a): a C-ABI CUDA library
(``include/pa.h``, built into ``_build/libpa.so``) and its PyTorch binding.

    from paged_kv_cache_193_gb300 import api
    out = api.decode(q, k_cache, v_cache, block_tables, context_lens, partition_size=512)

``workloads`` holds the seeded synthetic inputs used by the tests and the
benchmark.
"""
__all__ = ["api", "workloads", "build"]
