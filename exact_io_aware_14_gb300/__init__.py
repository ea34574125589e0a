"""GB300-native exact attention forward (sm_103a).

The compute lives in a C-ABI CUDA library (``libattn_sm103.so``, declared in
``include/attn.h``); ``_native`` only marshals arguments to it.
"""
from ._native import (  # noqa: F401
    ATTN_OK,
    AttnError,
    attn_fwd,
    attn_fwd_splitkv,
    attn_get_device_status,
    attn_splitkv_workspace_size,
    decode,
    forward,
    status_string,
)
