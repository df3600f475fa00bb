"""Batch-invariant decoder forward for GB300 (sm_103a).

The compute path is the C-ABI library libbi.so (include/bi.h) built from
csrc/*.cu; `_lib` is its thin ctypes binding (same entry-point names) and
`decoder` sequences the rollout and recompute calls.  Importing this package
does not load the library; the first call does, and fails loudly if it has not
been built.
"""
from . import _lib  # noqa: F401
from ._lib import *  # noqa: F401,F403

__all__ = [n for n in dir(_lib) if n.startswith(("bi_", "BI_"))] + ["BiError", "load"]
