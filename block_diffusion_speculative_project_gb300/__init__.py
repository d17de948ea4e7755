"""GB300-native one-pass block-diffusion draft step (DFlash / DFlow relay / DFlash 2).

The compute path is libdflash.so (hand-written sm_103a CUDA behind a C ABI, see
include/dflash.h); ``dflash`` is its ctypes binding and ``drafter.Drafter`` a holder
for one handle's device buffers. Importing ``dflash`` fails loudly when the library
has not been built.
"""
__all__ = ["dflash", "drafter", "build"]
