"""GB300 (sm_103a) fused Mixture-of-Experts layer forward.

The compute path is the CUDA library ``_build/libmoe_gb300.so`` (C ABI in
include/moe.h); this package is its ctypes binding (``_lib``, the C names)
plus a layer helper (``MoELayer``). There is no CPU fallback: the first use
of any binding name raises ImportError when the library is not built.
``mixture_experts_layer_15_gb300.build`` compiles it.
"""
import importlib

_SUBMODULES = ("build", "layer", "_lib")


def __getattr__(name):
    if name in _SUBMODULES:
        return importlib.import_module(f"{__name__}.{name}")
    if name in ("MoELayer", "Buffers"):
        return getattr(importlib.import_module(f"{__name__}.layer"), name)
    lib = importlib.import_module(f"{__name__}._lib")   # ImportError if the library is missing
    try:
        return getattr(lib, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
