"""GB300-native mixed-dtype FSDP communication-buffer packing.

The product is the C-ABI library built from ``csrc/`` (declared in
``include/fsdp_pack.h``); ``fsdp_pack`` is its thin Python binding and
``workloads`` the seeded synthetic layouts used by tests and benchmarks.
Importing the binding fails loudly when the library has not been built.
"""
import importlib

__all__ = ["fsdp_pack", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
