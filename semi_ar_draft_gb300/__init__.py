"""semi_ar_draft_gb300: the DSpark vocabulary-wide hot path on GB300 (sm_103a).

libdspark (CUDA, C ABI in include/dspark.h) runs every step; this package holds its build
script, its ctypes binding (`binding`, same names as the C entry points), allocation helpers
(`api`) and the seeded synthetic workloads (`workloads`).  The binding is imported lazily so
that the workloads module can be used without the compiled library.
"""

__all__ = ["binding", "api", "workloads", "build"]


def __getattr__(name):
    import importlib

    if name in __all__:
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
