"""Routed int4 mixture-of-experts layer for GB300 (sm_103a).

The compute runs in ``libmoe.so`` (C ABI in ``include/moe.h``); this package is
the Python binding.  The library is loaded on first use of any binding name
and that use raises ImportError when the library has not been built (there is
no fallback).  ``int4_routed_expert_fp32_gb300.build`` compiles it.
"""
import importlib

_BINDING = ("MoeConfig", "MoeError", "MoeLayer", "MoeWeights", "check_error", "combine",
            "dispatch", "dispatch_noalloc", "expert_ffn", "int4_linear", "int4_linear_partials",
            "int4_linear_stall_selftest", "int4_linear_int16", "quantize_rows_int16",
            "last_cuda_error", "launch_count",
            "lib", "linear_bf16", "quantize_int4", "quantize_int8",
            "quantize_rows", "set_tc_pair", "shared_expert",
            "rmsnorm", "route", "router_prepare", "status_string", "wait_selftest", "capi")


def __getattr__(name):
    if name in _BINDING:
        capi = importlib.import_module(".capi", __name__)
        return capi if name == "capi" else getattr(capi, name)
    raise AttributeError(name)


def __dir__():
    return sorted(list(globals()) + list(_BINDING))
