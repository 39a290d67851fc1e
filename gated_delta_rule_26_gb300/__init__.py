"""GB300-native (sm_103a) Kimi Delta Attention forward.

The compute lives in hand-written CUDA kernels behind the C-ABI library
``libkda`` (declared in ``include/kda.h``).  ``gated_delta_rule_26_gb300.kda``
is the thin Python binding over it (argument marshalling only); the library is
loaded on first use and a missing build raises instead of falling back to any
other implementation.
"""
import importlib

__all__ = ["kda", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
