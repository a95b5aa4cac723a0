"""Exact, IO-aware attention forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa_gb300.so`` built from
``csrc/``; ``fa.py`` is its ctypes binding.  Importing this package does not
load the library; the first call into ``fa`` does, and raises if it is
missing (there is no CPU fallback).
"""

import importlib

from . import workloads  # noqa: F401


def __getattr__(name):
    if name == "fwd":
        return importlib.import_module(".fa", __name__).fwd
    raise AttributeError(name)
