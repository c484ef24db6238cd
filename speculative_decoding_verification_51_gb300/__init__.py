"""GB300-native batched speculative-sampling verifier.

The compute path is a C-ABI CUDA library (``csrc/``, declared in
``include/spec_verify.h``) built for sm_103a; ``binding`` marshals arguments
to it with ctypes.  Importing the package loads nothing; the first call
through ``binding`` loads the library and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
