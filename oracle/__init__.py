"""CPU oracle for the CSA2 FP4 compressed-KV decode path.

TEST INFRASTRUCTURE, not part of the product. Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import this package. It is plain numpy, shares no
code with the CUDA path and imports nothing from it.

Modules:
  formats -- E2M1, E4M3 (fn) and E8M0 from their definitions.
  csa2    -- the method: merge, quantise/pack, append, indexer scores, Top-k,
             hierarchical pool, sparse attention with sliding window, the
             Full/Reindex/Reuse layer schedule, and the footprint arithmetic.

Parity status: every function is pinned by tests under ``tests/`` against page
numbers, format definitions, library routines, closed forms or brute force; no
function is unpinned.
"""
from . import formats, csa2  # noqa: F401
