"""Routed int4 mixture-of-experts layer for GB300 (sm_103a).

The compute runs in ``libmoe.so`` (C ABI in ``include/moe.h``); this package is
the Python binding.  Importing it fails when the library has not been built.
"""
from .capi import (MoeConfig, MoeError, MoeLayer, MoeWeights, check_error, combine, dispatch,  # noqa: F401
                   expert_ffn, int4_linear, lib, linear_bf16, quantize_rows, rmsnorm, route,
                   status_string, wait_selftest)
from .build import LIB_PATH  # noqa: F401
