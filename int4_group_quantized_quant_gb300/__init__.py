"""int4 weight-only group-quantized matvec for GB300 (sm_103a).

The compute lives in ``libgq4.so`` (hand-written CUDA kernels behind a C ABI,
declared in ``include/gq4.h``).  ``gq4`` is the thin Python binding over that
ABI; ``inputs`` draws seeded synthetic workloads.  Importing this package does
not load the CUDA library: ``from int4_group_quantized_quant_gb300 import gq4``
does, and fails loudly if the library has not been built.
"""

__all__ = ["gq4", "inputs", "build"]
