"""GB300-native Invariant Bit Packing (IBP).

``host_transfer_gb300.ibp`` binds the CUDA library ``libibp.so`` (built from
``csrc/`` by ``host_transfer_gb300.build``); ``host_transfer_gb300.workloads``
draws the seeded synthetic tables the tests and the benchmark use.  The
library is loaded on first use and there is no CPU fallback: a missing
``libibp.so`` is an error.
"""

__all__ = ["ibp", "workloads", "build"]
