"""moecache: a routed Mixture-of-Experts layer served from one GPU-resident
expert cache shared by all layers (GB300, sm_103a).

The compute path is the CUDA library ``_lib/libmoecache.so`` (C ABI in
``include/moecache.h``); ``moecache`` is its ctypes binding and is loaded on
first attribute access, so ``import expert_cache_serving_gb300.build`` works
before the library exists.
"""

__all__ = ["moecache"]


def __getattr__(name):
    if name == "moecache":
        import importlib

        return importlib.import_module(__name__ + ".moecache")
    raise AttributeError(name)
