"""GB300 (sm_103a) decode projection: y[B,N] = BF16(x[B,K] . W[N,K]^T).

The skinny BF16 linear a decode step applies at tensor-parallel degree 1
(runtime.dep page, DepProjection), as a C-ABI library of hand-written CUDA
kernels with a thin ctypes binding.  Submodules:

  _binding  the C functions under their C names, and ``Projection``
  synth     seeded synthetic inputs shared by tests, benchmark and oracle checks
  build     nvcc build of the library

The binding loads the library lazily, on first use, and raises if it is
missing: there is no CPU or library fallback.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import DepError, Projection, dep_tactic_t, lib, EXPORTS  # noqa: F401
