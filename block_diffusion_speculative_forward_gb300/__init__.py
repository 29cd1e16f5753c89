"""GB300 (sm_103a) propose forward of a block-diffusion draft head.

The compute path is libdflash.so (hand-written CUDA kernels behind the C ABI
of include/dflash.h); `binding` is its ctypes binding and `synthetic` draws
the seeded inputs. Importing the package loads nothing; the binding loads the
library on first use and raises if it is not built.
"""
__all__ = ["binding", "synthetic"]
