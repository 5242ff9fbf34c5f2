"""GB300 (sm_103a) grouped-convolution backward-weight (wgrad) as an implicit GEMM.

The compute path is the C-ABI library ``libwgrad.so`` built from ``csrc/``; the
Python module ``binding`` marshals arguments into it.  Importing this package
does not load the library; the first call into ``binding`` does, and raises if
it is missing.
"""
from . import synth  # noqa: F401

__all__ = ["synth"]
