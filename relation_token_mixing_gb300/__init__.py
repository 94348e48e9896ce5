"""Full Relation (Self-Exchange / Multi-Head Relation) operator for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library built from ``csrc/`` (see
``include/relation.h``); ``binding`` is its thin Python binding and
``inputs`` the seeded synthetic input generator.  Importing the package does
not load the CUDA library; the first binding call does.
"""

__all__ = ["binding", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
