"""GB300 implicit-GEMM convolution forward: Python binding of the C-ABI library.

The binding only marshals arguments; every step of the forward pass runs in the
CUDA library ``libconvfwd.so`` built from ``csrc/``.  Loading is lazy: importing
the package never needs a GPU, but the first call fails loudly if the library
has not been built.
"""
from .binding import *  # noqa: F401,F403
