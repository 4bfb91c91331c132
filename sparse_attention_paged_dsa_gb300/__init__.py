"""GB300-native decode-step DSA indexer: paged C4 index keys -> scores -> top-k.

The compute path lives in the CUDA library ``libdsa_indexer.so`` built from
``csrc/`` for sm_103a; ``binding`` is its thin Python front-end (argument
marshalling only).  ``inputs`` draws seeded synthetic workloads.  Nothing in
this package computes indexer results on the CPU.
"""

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in ("binding", "inputs"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
