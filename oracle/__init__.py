"""fp64 CPU oracle -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports it, and it imports nothing from the product.

Contents
  attention.py  exact softmax attention over a paged cache (C, fp64, OpenMP)
                plus the partial-state / merge definition of split-KV decoding
  streamk.py    the Stream-K one-wave work split, a round-robin queue fill and a
                greedy list-scheduling simulator (integer work, exact)

Every function is pinned by tests under ``tests/test_oracle_*.py`` against
closed forms, invariants, a library routine (torch SDPA in fp64) and the worked
examples printed on the pages (``tests/golden/``).
"""
