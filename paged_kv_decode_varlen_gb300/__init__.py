"""Paged varlen attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpa.so`` built from ``csrc/``
(declared in ``include/pa.h``); ``binding`` marshals torch tensors into it.
``workloads`` builds seeded synthetic batches.  Importing this package does
not load the library; importing ``binding`` does, and raises if the library
is missing.
"""
from . import workloads  # noqa: F401  (numpy only)
