"""Exact, IO-aware attention forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libfa_gb300.so`` built from
``csrc/``; ``fa.py`` is its ctypes binding.  Importing this package does not
load the library; the first call into ``fa`` does, and raises if it is
missing (there is no CPU fallback).
"""

from . import workloads  # noqa: F401


def __getattr__(name):
    if name in ("fwd", "fa"):
        from . import fa as _fa
        return _fa if name == "fa" else _fa.fwd
    raise AttributeError(name)
