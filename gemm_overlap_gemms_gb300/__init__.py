"""Active-shape tensor-parallel AG-GEMM / GEMM-RS for one GB300 (sm_103a).

The compute path lives in the C-ABI library ``libubgemm.so`` (CUDA kernels plus host
orchestration, built from ``csrc/``); ``ub`` is its thin ctypes binding and ``synth``
holds the seeded workload generators. Importing this package loads nothing native;
the first call into ``ub`` loads the library and raises if it is missing.
"""
__all__ = ["ub", "synth"]
