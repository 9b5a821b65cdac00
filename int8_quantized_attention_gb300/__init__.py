"""GB300-native INT8-QK quantized attention (SageAttention-style).

The compute path is the C-ABI library ``libsageattn.so`` built from
``csrc/`` for sm_103a; :mod:`.binding` marshals torch tensors into its
entry points.  Submodules are imported lazily so that the seeded input
generators in :mod:`.workloads` stay usable on machines without a GPU.
"""
import importlib

__all__ = ["binding", "build", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
