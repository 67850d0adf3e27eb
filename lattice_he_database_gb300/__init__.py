"""GB300-native server-side scan of lattice-based single-server PIR.

RowSel (OnionPIR-family first fold) over an NTT-domain RNS database and the
scalar-HE (SimplePIR-family) byte-DB scan, as hand-written sm_103a CUDA
kernels behind the C ABI in include/pir.h.  ``pir`` is the thin binding.
"""
from .pir import *  # noqa: F401,F403
from . import pir  # noqa: F401
