"""GB300-native batched CTC prefix beam search.

The decoder itself is a C-ABI CUDA library (``csrc/``, declared in
``include/ctcpb.h``); this package holds its thin ctypes binding and the seeded
input generators.  Importing it does not load the library: the first decoder
call does, and fails loudly if the library is missing.
"""
__all__ = ["synth"]
