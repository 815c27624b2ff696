"""paged_kv_decode_splitk_gb300 -- paged-decode split-K attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libpd.so`` built from ``csrc/``; the
Python side (``pd``) only marshals arguments into it.  Importing this package
does not load the library: the first call does, and it raises if the library
is missing.  There is no CPU fallback.
"""

__all__ = ["pd", "workloads"]
