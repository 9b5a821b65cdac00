"""GB300-native INT8-QK quantized attention (SageAttention-style).

The compute path is the C-ABI library ``libsageattn.so`` built from
``csrc/`` for sm_103a; :mod:`.binding` marshals torch tensors into its
entry points.  The binding is imported lazily so that the seeded input
generators in :mod:`.workloads` stay usable on machines without a GPU.
"""
__all__ = ["binding", "workloads"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    if name == "workloads":
        from . import workloads
        return workloads
    raise AttributeError(name)
