"""GB300-native scaled casts of training tensors to OCP FP8.

  fp8q        ctypes binding of libfp8q.so (the sm_103a kernels)
  build       nvcc build of libfp8q.so
  synthetic   seeded input generators for the workloads (no arithmetic of
              the method)

Nothing is loaded at import time; ``fp8q.load()`` opens the library.
"""
__all__ = ["fp8q", "build", "synthetic"]
