"""Epoch routed-expert MoE layer iteration for GB300 (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (see
``include/epoch.h``); this package holds its ctypes binding (``binding``), a
torch-facing wrapper (``layer.EpochLayer``) and the in-tree build
(``builder.build``). Importing the package does not load the library; the first
call into it does, and fails loudly if the library has not been built.
"""
__all__ = ["binding", "builder", "layer"]


def __getattr__(name):
    if name in ("binding", "builder", "layer"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    if name in ("EpochLayer", "payload_to_torch"):
        from . import layer as _layer
        return getattr(_layer, name)
    raise AttributeError(name)
