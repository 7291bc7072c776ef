"""CPU float64 oracle of the decoder-only Transformer forward pass.

Test infrastructure only: the test suite, the package smoke check and the
benchmark's CPU-baseline leg may use it; the product path never does.
"""
from .ref import *  # noqa: F401,F403
from . import ref  # noqa: F401
