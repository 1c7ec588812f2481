"""GB300-native batched speculative-sampling verify step.

The compute lives in a C-ABI shared library of hand-written CUDA kernels for
sm_103a (``csrc/``, declared in ``include/spec_verify.h``).  ``binding`` is a
thin ctypes layer over it with the same entry-point names; ``workloads`` draws
seeded synthetic inputs.  Importing the package loads nothing: the library is
loaded (and built if missing) on the first call into ``binding``.
"""
__all__ = ["binding", "workloads"]
