"""fp64 CPU oracle for the LOCKS decode hot path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import or run it.  It shares no code, tables or
constants with the CUDA library under ``sparse_long_context_locks_gb300/``.

Source of the method: "LOCKS: Page-Local Compact Key Summaries for Efficient
Long-Context Decoding" (J. Hwang, arXiv 2607.24555) -- the technical summary's
§2 "Method" (page-local spectral decomposition, quantisation, reconstruction
and selection, group-shared selection) and the paper abstract.

Parity status per function is listed in ``oracle/locks_oracle.py``'s header.
"""

from .locks_oracle import *  # noqa: F401,F403
