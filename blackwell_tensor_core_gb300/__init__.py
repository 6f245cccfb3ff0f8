"""GB300-native half-precision GEMM library (sm_103a, tcgen05/TMA kernels).

The compute path is the C-ABI shared library ``libbwgemm.so`` built from
``csrc/``; ``ops`` is its thin Python binding (argument marshalling only).
Importing this package loads nothing: the library is loaded on first use and
a missing or unbuilt library raises instead of falling back to anything else.
"""

__all__ = ["ops", "workloads"]
