"""Oracle for the paged KV-cache decode path: plain, slow, obviously correct.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) may import,
call or load anything in this package.  It shares no code with the CUDA
library under ``paged_kv_cache_227_gb300/`` and never imports it.

Contents
  attention   fp64 paged decode attention (C, ``paged_attention.c``), the
              plain definition "gather through the block table, then
              softmax(scale * K q) V" ("Serving", section 23.4 Paged Attention;
              "The KV Cache" teaser: the cache is exact).
  cache       byte-level models of the cache write and the copy-on-write block
              copy, and the KV-size closed form of "Serving" section 23.1.
  allocator   a reference block allocator (free list, reference counts, fork,
              copy-on-write) in plain Python.

Every function here is pinned by tests that check it against something other
than itself (a library routine, a closed form, the pages' printed numbers, an
invariant, brute force on tiny inputs); see ``tests/test_oracle_*.py``.
"""
from .attention import build, paged_decode, fp16_bits_to_double, bf16_bits_to_double, max_threads  # noqa: F401
from . import cache, allocator  # noqa: F401
