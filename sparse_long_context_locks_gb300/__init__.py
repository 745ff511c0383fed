"""LOCKS sparse long-context decode for GB300 (sm_103a).

The product is the C-ABI library ``liblocks.so`` built from ``csrc/`` (entry
points declared in ``include/locks.h``); ``locks`` is its thin ctypes binding
and ``workload`` draws seeded synthetic inputs.  Importing the package loads
nothing: the binding loads the library on first use and raises if it is
missing (there is no CPU fallback).
"""

__all__ = ["locks", "workload", "build"]
