"""ctypes declarations of libls (the C ABI in ``include/ls.h``).

Loading fails loudly when the library has not been built: there is no other
implementation of the decode step in this package.
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libls.so")

LS_OK = 0
LS_ERR_INVALID = -1
LS_ERR_ALIGN = -2
LS_ERR_SLOT = -3
LS_ERR_CUDA = -4
LS_ERR_SIZE = -5

LS_DEV_SLOT_RANGE = 1
LS_DEV_TIMEOUT = 2
LS_DEV_BAD_STATE = 4
LS_DEV_SLOT_DUP = 8

LS_EAGER_FP32 = 0
LS_DEFERRED_FP32 = 1
LS_WINDOW_INT8 = 2

LS_GATE_SCALAR = 0
LS_GATE_PER_KEY = 1

LS_MAX_WINDOW = 256
LS_INT8_COLUMN_SCALES = 1
LS_MAX_COMPENSATORS = 8
LS_PLAIN_UPDATE = 1 << 12
LS_LOG_BF16_K = 1 << 13
LS_INT8_FP16_RECORDS = 1 << 14
LS_CHECK_SLOTS = 1 << 15
LS_SPLIT_STATIC_SCRATCH_BYTES = 16 << 20


def LS_INT8_COMPENSATORS(r: int) -> int:
    return int(r) << 8
LS_ABI_VERSION = 5  # the include/ls.h these prototypes follow

# Every symbol include/ls.h declares.
EXPORTS = (
    "ls_error_string", "ls_abi_version", "ls_pool_required_bytes", "ls_pool_create",
    "ls_pool_destroy", "ls_pool_load", "ls_pool_reset_slots", "ls_decode_step",
    "ls_decode_step_split", "ls_split_scratch_bytes", "ls_decode_step_split_static",
    "ls_step_staging_bytes", "ls_decode_step_host", "ls_window_commit", "ls_pool_read",
    "ls_pool_read_int8", "ls_pool_read_int8_col_scales", "ls_pool_read_compensators",
    "ls_pool_read_log_meta",
    "ls_pool_status",
)


class LsDesc(C.Structure):
    _fields_ = [("num_slots", C.c_int32), ("num_heads", C.c_int32), ("d_k", C.c_int32),
                ("d_v", C.c_int32), ("variant", C.c_int32), ("gate", C.c_int32),
                ("window", C.c_int32), ("flags", C.c_uint32)]


class LsError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})")


_lib = None


def load() -> C.CDLL:
    """Load libls.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libls.so is not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(LIB_PATH)
    P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
    sig = {
        "ls_error_string": (C.c_char_p, [C.c_int]),
        "ls_abi_version": (C.c_int, []),
        "ls_pool_required_bytes": (C.c_int, [C.POINTER(LsDesc), C.POINTER(SZ)]),
        "ls_pool_create": (C.c_int, [C.POINTER(LsDesc), P, SZ, P, C.POINTER(P)]),
        "ls_pool_destroy": (C.c_int, [P]),
        "ls_pool_load": (C.c_int, [P, P, I32, P, P]),
        "ls_pool_reset_slots": (C.c_int, [P, P, I32, P]),
        "ls_decode_step": (C.c_int, [P, P, I32, P, P, P, P, P, P, P]),
        "ls_step_staging_bytes": (C.c_int, [P, I32, C.POINTER(SZ)]),
        "ls_decode_step_split": (C.c_int, [P, P, I32, P, P, P, P, P, P, P, SZ, P]),
        "ls_split_scratch_bytes": (C.c_int, [P, I32, C.POINTER(SZ)]),
        "ls_decode_step_split_static": (C.c_int, [P, P, I32, P, P, P, P, P, P, P]),
        "ls_decode_step_host": (C.c_int, [P, P, I32, P, P, P, P, P, P, P, SZ, P]),
        "ls_window_commit": (C.c_int, [P, P, I32, P]),
        "ls_pool_read": (C.c_int, [P, P, I32, P, P]),
        "ls_pool_read_int8": (C.c_int, [P, P, I32, P, P, P]),
        "ls_pool_read_int8_col_scales": (C.c_int, [P, P, I32, P, P]),
        "ls_pool_read_compensators": (C.c_int, [P, P, I32, P, P, P]),
        "ls_pool_read_log_meta": (C.c_int, [P, P, I32, P, P, P]),
        "ls_pool_status": (C.c_int, [P, P, C.POINTER(I32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.ls_abi_version() != LS_ABI_VERSION:
        raise ImportError(f"libls.so has ABI version {lib.ls_abi_version()}, the binding "
                          f"expects {LS_ABI_VERSION}: rebuild it")
    _lib = lib
    return lib


def error_string(code: int) -> str:
    try:
        return load().ls_error_string(int(code)).decode()
    except ImportError:
        return f"status {code}"


def check(code: int, what: str) -> None:
    if code != LS_OK:
        raise LsError(code, what)
