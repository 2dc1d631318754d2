"""B300-native forward pass (prefill + KV-cache decode) of a nanochat-style GPT.

The compute lives in ``libnc.so`` (hand-written sm_103a CUDA kernels behind the
C ABI of ``include/nc.h``); ``nc.py`` is a ctypes binding over it.
"""
from .nc import (  # noqa: F401
    Model, NcConfig, NcError, make_config, lib, header_functions, LIB_PATH, NC_BF16, NC_F32,
)
