"""Zero-SM collective schedules over k simulated ranks on one GB300.

The compute path is libhoc.so (CUDA kernels for sm_103a plus a C++ runtime
behind the C ABI in include/hoc.h); ``hoc`` is its ctypes binding and
``inputs`` the seeded synthetic workloads.
"""
from . import hoc  # noqa: F401
from .hoc import Comm, Config, HocError  # noqa: F401

__all__ = ["hoc", "Comm", "Config", "HocError"]
