"""GB300-native MoE-layer forward: a persistent megakernel behind a C ABI.

The compute path is the CUDA library ``_build/libmoe.so`` (built from
``csrc/`` for sm_103a); this package only marshals arguments to it.  There is
no fallback: importing the binding raises if the library is missing.
"""
from .binding import (  # noqa: F401
    MOE_OK, MOE_E_INVAL, MOE_E_CUDA, MOE_E_TIMEOUT, MOE_E_DEVICE, MOE_E_NOMEM, MOE_E_STATE,
    MOE_MODE_PERSISTENT, MOE_MODE_MULTIKERNEL, MOE_MODE_STATIC, OPTIONS, STATS, MoEError, MoELayer, lib,
    header_symbols, load_library,
)
