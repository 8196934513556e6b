"""GB300-native (sm_103a) Lizard hybrid token mixer.

The compute lives in liblizard.so (C ABI declared in include/lizard.h, kernels in
csrc/); `lizard` is its thin Python binding and `inputs` the seeded synthetic
input generator.  Importing the package does not load the library; the first
call into `lizard` does, and raises if it has not been built.
"""
__all__ = ["inputs", "lizard"]
