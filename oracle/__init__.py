"""fp64 CPU oracle of the MoE expert layer — TEST INFRASTRUCTURE ONLY.

Imported only by ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg (``bench.py --impl reference`` and the ``cpu_baseline`` field).
The CUDA library and its Python binding never import it and share no code,
tables or helpers with it; the two meet only in the seeded input generators
(``token_dispatch_grouped_router_gb300.workloads``), which hold none of the
layer's arithmetic.

Every function is pinned by ``tests/test_oracle_*.py`` against brute force,
closed forms, library routines or finite differences.  The end-to-end layer
numbers cannot be pinned to the pages, which print no layer output for this
path (parity unpinned at that level; each step below it is pinned).
"""
from . import layer, mxfp8, padded  # noqa: F401
from .layer import *  # noqa: F401,F403
