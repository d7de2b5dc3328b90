"""Batch-1 quantized Llama decode step for NVIDIA GB300 (sm_103a).

The compute lives in ``libnt.so`` (CUDA, built from ``csrc/``); ``nt`` is the
ctypes binding of its C ABI (``include/nt.h``) and ``workloads`` the model and
sweep definitions.
"""
from . import nt, workloads  # noqa: F401
from .nt import *  # noqa: F401,F403
