"""GB300-native DFlash draft step, greedy verify-accept and draft-KV commit.

The compute lives in libdflash.so (hand-written sm_103a CUDA behind a C ABI,
declared in include/dflash.h).  This package is a thin ctypes binding over it
(`api`), the workload shapes (`configs`) and the seeded synthetic input
generators (`synth`).  Importing the package does not load the library; the
first call into `api` does, and fails loudly when it is missing.
"""
__all__ = ["api", "configs", "synth"]
