"""GB300-native decoder-only forward pass over a KV cache.

The compute path is ``libdec.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/dec.h``); ``decoder_only_forward_gb300.dec`` is its thin
ctypes binding.  Importing this package loads nothing: the binding loads the
library on first import and raises if it is missing.
"""
