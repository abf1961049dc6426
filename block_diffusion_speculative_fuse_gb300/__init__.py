"""GB300-native DFlash-style block-diffusion drafting: C-ABI CUDA library
(``include/dflash.h``, ``csrc/``) with a thin ctypes binding.

Importing the package does not load the library; ``binding.load()`` (called
by every binding function) does, and raises if it has not been built.
"""
from . import _build  # noqa: F401

__all__ = ["binding", "device", "_build"]
