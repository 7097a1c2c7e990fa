"""GB300-native depth-routing read of attention residuals.

The compute lives in ``libattnres_gb300.so`` (CUDA kernels for sm_103a behind
the C ABI of ``include/attnres.h``); ``binding`` is its ctypes mirror and
``workload`` drives a whole microbatch (appends, every site's forward, every
site's backward in reverse) through it. Importing ``binding`` (or any name it
exports, through this package) fails loudly when the library is not built.
"""

__all__ = ["binding", "build", "workload"]


def __getattr__(name):
    import importlib
    if name in ("binding", "build", "workload"):
        return importlib.import_module(f"{__name__}.{name}")
    b = importlib.import_module(f"{__name__}.binding")
    if hasattr(b, name):
        return getattr(b, name)
    raise AttributeError(name)
