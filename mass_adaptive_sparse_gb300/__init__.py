"""MassAlloc Attention (MALA) for GB300 (sm_103a).

The compute lives in ``libmala.so`` (CUDA kernels behind a C ABI, declared in
``include/mala.h``); :mod:`.api` is a thin ctypes binding with the same names.
:mod:`.synthetic` draws the seeded planted-peak inputs.  Importing the package
does not load the CUDA library; the first call into :mod:`.api` does, and
fails loudly if it is missing.
"""
__all__ = ["api", "synthetic"]
