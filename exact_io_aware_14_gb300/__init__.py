"""GB300-native exact attention forward (sm_103a).

The compute lives in a C-ABI CUDA library (``libattn_sm103.so``, declared in
``include/attn.h``); this package only marshals arguments to it.
"""
