"""GB300-native renderer bank attention (FlashForward in-flight KV bank).

The compute path is libff.so (hand-written sm_103a kernels behind a C ABI,
declared in include/ff.h); ``ff`` is its ctypes binding and ``synth`` the
seeded input generator.  Importing the package loads nothing: the binding
loads the library on first use and raises if it has not been built.
"""
__all__ = ["ff", "synth", "build"]
