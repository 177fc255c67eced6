"""Float64 CPU oracle for the group-quantized weight-only GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package: only the
test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA path (no kernels, headers,
helpers or tables); the only module both sides use is ``gq_synth``, the seeded input
generator, which holds none of the method's arithmetic.

Every function here is pinned by a ``-m "not gpu"`` test against something other than
itself (values the pages print, closed forms, library special cases, brute force on tiny
inputs).  Parity unpinned: none.
"""
from .gq_oracle import *  # noqa: F401,F403
