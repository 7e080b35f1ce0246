"""fp64 CPU oracle for MassAlloc Attention.  Test infrastructure only: the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg are the
only callers; the product path never imports it."""
from .mala_oracle import *  # noqa: F401,F403
