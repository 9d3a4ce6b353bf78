"""GB300-native fused quantized LM-head (vocab-blocked Flash Cut-Cross-Entropy).

The compute path is a C-ABI CUDA library (``libqhead.so``, declared in
``include/qhead.h``); :mod:`verify_vocab_blocked_gb300.qhead` is its thin
ctypes binding.  Importing this package loads nothing; the first call into the
binding loads the library and fails loudly if it has not been built.
"""
