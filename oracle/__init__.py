"""TEST INFRASTRUCTURE ONLY: the CPU oracle for the paged KV-cache hot path.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import, call, link or execute anything in this package.  The
product path (``paged_kv_cache_138_gb300``) never imports it, and this package
never imports the product: the two share no kernels, headers, helpers, tables or
pre/post-processing.  Inputs reach both sides from the seeded generators in
``paged_kv_cache_138_gb300.workloads``, which hold none of the method's
arithmetic.

Contents
  attention.py      fp64 paged decode attention (C, OpenMP) + a NumPy dense form
  cache_ops.py      slot mapping, reshape_and_cache and copy_blocks definitions
  block_manager.py  the BlockManager of "P06 BlockManager" (free list, ref counts,
                    chained-hash prefix cache, LRU evictable pool, atomicity),
                    with fork + copy-on-write from "ans20xx day 31"

Parity status: every function here is pinned by ``-m "not gpu"`` tests against
values the pages print or fix (worked examples, closed forms, invariants, library
routines); none is "parity unpinned".
"""
