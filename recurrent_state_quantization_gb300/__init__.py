"""GB300-native decode step of delta-rule linear attention over a state pool.

Three storage variants of the recurrent state behind one C ABI (``libls``):
eager FP32, deferred base + log (DeltaLog), and per-window INT8 (LeapQuant).
The native library is loaded on first use and must have been built
(``__graft_entry__.build()``); there is no fallback implementation.
"""
from ._native import (LsError, LS_DEV_BAD_STATE, LS_DEV_SLOT_DUP, LS_DEV_SLOT_RANGE,  # noqa: F401
                      LS_DEV_TIMEOUT)
from .pool import StatePool, required_bytes  # noqa: F401

__all__ = ["StatePool", "required_bytes", "LsError", "LS_DEV_SLOT_RANGE", "LS_DEV_TIMEOUT",
           "LS_DEV_BAD_STATE", "LS_DEV_SLOT_DUP"]
