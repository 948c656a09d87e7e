"""GB300-native paged KV cache: paged decode attention, reshape_and_cache and
copy_blocks as hand-written sm_103a CUDA kernels behind a C ABI (libpagedkv),
plus the host BlockManager that produces block tables and slot mappings.

Import ``paged_kv_cache_138_gb300.ops`` for the kernels and
``paged_kv_cache_138_gb300.block_manager`` for the host manager; both load
``libpagedkv.so`` and raise if it has not been built.
"""
__all__ = ["ops", "block_manager", "workloads", "accounting", "build"]
