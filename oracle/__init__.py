"""CPU oracle -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports, links or calls anything under ``oracle/``.
"""
