"""Gated DeltaNet chunked forward for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libgdn.so`` built from ``csrc/``;
``gdn`` is its thin ctypes binding (argument marshalling only).
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]
