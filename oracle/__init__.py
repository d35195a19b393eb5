"""fp64 CPU oracle for Kimi Delta Attention.  TEST INFRASTRUCTURE ONLY.

Two independent codings of the same definition (Kimi K3 technical report,
section 2.1.1, Eq. 1 and Eq. 5): ``numpy_ref`` (NumPy, small cases, plus the
chunkwise form of Eq. 3-4 and the segment maps of Eq. 17) and ``c_ref``
(plain C with OpenMP, for workload-sized samples and the CPU baseline).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library.
"""
from . import numpy_ref  # noqa: F401
from . import c_ref  # noqa: F401
