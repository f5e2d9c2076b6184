"""kev: packed, question-isolated attention for one GB300 (sm_103a).

The compute path is libkev.so (CUDA kernels behind the C ABI in include/kev.h);
``binding`` is its ctypes binding with the same entry-point names.  The
binding is loaded on first use of a ``kev_*`` name and raises ImportError if
the library has not been built -- there is no fallback.
"""
from __future__ import annotations

import importlib


def __getattr__(name):
    if name.startswith("kev_") or name in ("KevError", "make_shape", "library_path", "binding"):
        mod = importlib.import_module(".binding", __name__)
        return mod if name == "binding" else getattr(mod, name)
    raise AttributeError(name)
