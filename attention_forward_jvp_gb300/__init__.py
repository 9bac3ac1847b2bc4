"""Fused attention forward + JVP for GB300 (sm_103a).

The compute path is the C-ABI library ``libattn_jvp.so`` built from
``csrc/``; :mod:`.binding` is the thin ctypes layer above it.  Importing the
package loads nothing: the library is opened on first use and a missing
library raises immediately (there is no CPU fallback).
"""
__all__ = ["binding", "workloads"]
