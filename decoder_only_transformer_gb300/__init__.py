"""GB300-native forward pass of a pre-norm decoder-only Transformer LM.

The compute lives in ``libtfm.so`` (hand-written sm_103a CUDA kernels behind a
C ABI declared in ``include/tfm.h``); ``decoder_only_transformer_gb300.tfm``
is the thin ctypes binding.  Importing this package does not load the library;
the binding loads it on first use and raises if it is missing.
"""
__all__ = ["accounting", "tfm"]
