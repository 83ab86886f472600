"""Weight-only mixed-bit packed matvec for GB300 (sm_103a).

The computation lives in the CUDA library ``_lib/libqmv.so`` (sources in
``csrc/``, C ABI in ``include/qmv.h``); ``qmv`` is its ctypes binding and
``build`` compiles it.  Importing ``qmv`` raises if the library is missing.
"""
import importlib

__all__ = ["qmv", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
