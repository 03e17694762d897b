"""RLA-2 / RAPT causal ReLU linear attention for GB300 (sm_103a).

The compute path is the C-ABI library ``librapt.so`` (include/rapt.h) built from ``csrc/``;
``binding`` marshals torch tensors into it. Importing the package does not load the library:
the first call does, and raises if it is not built. ``synthetic`` holds the seeded input
generators.
"""

__all__ = ["rapt_prefill_fwd", "rapt_varlen_fwd", "rapt_decode_step", "rla_l2_fwd"]


def __getattr__(name):
    if name in __all__:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
