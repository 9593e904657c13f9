"""Python binding of libls: a pool of recurrent states in caller-owned HBM.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libls.so``; PyTorch provides the device memory and the stream.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import _native as N

VARIANTS = {"eager": N.LS_EAGER_FP32, "deferred": N.LS_DEFERRED_FP32, "int8": N.LS_WINDOW_INT8}
GATES = {"scalar": N.LS_GATE_SCALAR, "per_key": N.LS_GATE_PER_KEY}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _need(t: torch.Tensor, name: str, dtype, device, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _flags(col_scales: bool, compensators: int, plain: bool = False, k16: bool = False,
           r16: bool = False, check_slots: bool = False) -> int:
    return ((N.LS_INT8_COLUMN_SCALES if col_scales else 0) | N.LS_INT8_COMPENSATORS(compensators)
            | (N.LS_PLAIN_UPDATE if plain else 0) | (N.LS_LOG_BF16_K if k16 else 0)
            | (N.LS_INT8_FP16_RECORDS if r16 else 0) | (N.LS_CHECK_SLOTS if check_slots else 0))


def required_bytes(num_slots, num_heads, variant="eager", gate="scalar", window=0,
                   d_k=128, d_v=128, col_scales=False, compensators=0, plain=False,
                   k16=False, r16=False, check_slots=False) -> int:
    lib = N.load()
    d = N.LsDesc(num_slots, num_heads, d_k, d_v, VARIANTS[variant], GATES[gate], window,
                 _flags(col_scales, compensators, plain, k16, r16, check_slots))
    out = C.c_size_t(0)
    N.check(lib.ls_pool_required_bytes(C.byref(d), C.byref(out)), "ls_pool_required_bytes")
    return int(out.value)


class StatePool:
    """``num_slots`` x ``num_heads`` recurrent states of one layer on one GPU.

    variant: "eager" (dense FP32), "deferred" (FP32 base + log, merge interval
    ``window``) or "int8" (INT8 base, window ``window``).
    gate: "scalar" (Gated DeltaNet) or "per_key" (KDA).
    col_scales (int8): the smoothed per-value-column format (LeapQuant §3.4
    eq. 7, App. B.3) instead of one scale per key row.
    compensators (int8): r Compensator Tokens per window (LeapQuant §3.3).
    plain (eager / deferred): the update pair (k, v) without the delta-rule
    correction (DeltaLog Table 1: RWKV6 with the per-key gate, GLA, RetNet).
    k16 (deferred / int8): bfloat16 key-side log factors (DeltaLog §3.4).
    r16 (int8): the window's records (k, u) and compensator pairs in IEEE
    binary16 (LeapQuant §4.1, §4.3).
    check_slots: every call that changes states first checks on the device
    that its slot list repeats no slot, and flags LS_DEV_SLOT_DUP if it does
    (read by ``status()``); one extra launch per call.
    """

    def __init__(self, num_slots: int, num_heads: int, variant: str = "eager",
                 gate: str = "scalar", window: int = 0, d_k: int = 128, d_v: int = 128,
                 device=None, stream=None, col_scales: bool = False, compensators: int = 0,
                 plain: bool = False, k16: bool = False, r16: bool = False,
                 check_slots: bool = False):
        self.lib = N.load()
        self.variant, self.gate = variant, gate
        self.P, self.H, self.d_k, self.d_v = int(num_slots), int(num_heads), int(d_k), int(d_v)
        self.window = int(window)
        self.dl = 1 if gate == "scalar" else self.d_k
        dev = torch.device(device) if device is not None else torch.device("cuda")
        if dev.type != "cuda":
            raise ValueError("StatePool lives on a CUDA device")
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.col_scales = bool(col_scales)
        self.compensators = int(compensators)
        self.plain = bool(plain)
        self.k16 = bool(k16)
        self.r16 = bool(r16)
        self.check_slots = bool(check_slots)
        self.desc = N.LsDesc(self.P, self.H, self.d_k, self.d_v, VARIANTS[variant], GATES[gate],
                             self.window, _flags(self.col_scales, self.compensators, self.plain,
                                                 self.k16, self.r16, self.check_slots))
        nbytes = C.c_size_t(0)
        N.check(self.lib.ls_pool_required_bytes(C.byref(self.desc), C.byref(nbytes)),
                "ls_pool_required_bytes")
        self.nbytes = int(nbytes.value)
        with torch.cuda.device(self.device):
            self.mem = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=self.device)
        off = (-self.mem.data_ptr()) % 256
        self._mem_ptr = self.mem.data_ptr() + off
        handle = C.c_void_p()
        with torch.cuda.device(self.device):
            N.check(self.lib.ls_pool_create(C.byref(self.desc), C.c_void_p(self._mem_ptr),
                                            self.nbytes, C.c_void_p(_stream(stream)),
                                            C.byref(handle)), "ls_pool_create")
        self.handle = handle
        self._staging = None
        self._split_scratch = None

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            try:
                self.lib.ls_pool_destroy(h)
            except Exception:
                pass
            self.handle = None

    # ---- helpers ----------------------------------------------------------
    def _slots(self, slots) -> torch.Tensor:
        if not isinstance(slots, torch.Tensor):
            slots = torch.as_tensor(list(slots) if not isinstance(slots, range) else list(slots),
                                    dtype=torch.int32)
        if slots.dtype != torch.int32:
            slots = slots.to(torch.int32)
        return slots.to(self.device).contiguous()

    # ---- the C ABI calls ---------------------------------------------------
    def decode_step(self, slot_idx, q, k, v, log_decay, beta, y=None, stream=None):
        """One token for ``batch`` requests; returns y [batch, H, d_v]."""
        slot_idx = self._slots(slot_idx)
        B = int(slot_idx.numel())
        dev, f32 = self.device, torch.float32
        _need(q, "q", f32, dev, (B, self.H, self.d_k))
        _need(k, "k", f32, dev, (B, self.H, self.d_k))
        _need(v, "v", f32, dev, (B, self.H, self.d_v))
        _need(log_decay, "log_decay", f32, dev,
              (B, self.H) if self.dl == 1 else (B, self.H, self.d_k))
        _need(beta, "beta", f32, dev, (B, self.H))
        if y is None:
            y = torch.empty(B, self.H, self.d_v, dtype=f32, device=dev)
        _need(y, "y", f32, dev, (B, self.H, self.d_v))
        rc = self.lib.ls_decode_step(self.handle, _ptr(slot_idx), B, _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(log_decay), _ptr(beta), _ptr(y),
                                     C.c_void_p(_stream(stream)))
        N.check(rc, "ls_decode_step")
        return y

    def split_scratch_bytes(self, batch: int) -> int:
        out = C.c_size_t(0)
        N.check(self.lib.ls_split_scratch_bytes(self.handle, int(batch), C.byref(out)),
                "ls_split_scratch_bytes")
        return int(out.value)

    def decode_step_split(self, slot_idx, q, k, v, log_decay, beta, y=None, scratch=None,
                          stream=None):
        """ls_decode_step_split (deferred / INT8): the replay coefficients are
        computed into ``scratch`` (a uint8 device tensor of at least
        split_scratch_bytes(batch) bytes; one is kept on the pool when None)
        by a first kernel, then the step applies them.  Returns y."""
        slot_idx = self._slots(slot_idx)
        B = int(slot_idx.numel())
        dev, f32 = self.device, torch.float32
        _need(q, "q", f32, dev, (B, self.H, self.d_k))
        _need(k, "k", f32, dev, (B, self.H, self.d_k))
        _need(v, "v", f32, dev, (B, self.H, self.d_v))
        _need(log_decay, "log_decay", f32, dev,
              (B, self.H) if self.dl == 1 else (B, self.H, self.d_k))
        _need(beta, "beta", f32, dev, (B, self.H))
        if y is None:
            y = torch.empty(B, self.H, self.d_v, dtype=f32, device=dev)
        _need(y, "y", f32, dev, (B, self.H, self.d_v))
        need = self.split_scratch_bytes(B)
        if scratch is None:
            if self._split_scratch is None or self._split_scratch.numel() < need:
                self._split_scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
            scratch = self._split_scratch
        if scratch.device != dev or not scratch.is_contiguous():
            raise ValueError("scratch must be a contiguous tensor on the pool's device")
        rc = self.lib.ls_decode_step_split(self.handle, _ptr(slot_idx), B, _ptr(q), _ptr(k),
                                           _ptr(v), _ptr(log_decay), _ptr(beta), _ptr(y),
                                           _ptr(scratch), scratch.numel() * scratch.element_size(),
                                           C.c_void_p(_stream(stream)))
        N.check(rc, "ls_decode_step_split")
        return y

    def decode_step_split_static(self, slot_idx, q, k, v, log_decay, beta, y=None, stream=None):
        """ls_decode_step_split_static: the split-replay step with the
        library's fixed device scratch (allocates nothing).  Calls that may
        run concurrently on one device race on that scratch."""
        slot_idx = self._slots(slot_idx)
        B = int(slot_idx.numel())
        dev, f32 = self.device, torch.float32
        _need(q, "q", f32, dev, (B, self.H, self.d_k))
        _need(k, "k", f32, dev, (B, self.H, self.d_k))
        _need(v, "v", f32, dev, (B, self.H, self.d_v))
        _need(log_decay, "log_decay", f32, dev,
              (B, self.H) if self.dl == 1 else (B, self.H, self.d_k))
        _need(beta, "beta", f32, dev, (B, self.H))
        if y is None:
            y = torch.empty(B, self.H, self.d_v, dtype=f32, device=dev)
        _need(y, "y", f32, dev, (B, self.H, self.d_v))
        need = self.split_scratch_bytes(B)
        if need > N.LS_SPLIT_STATIC_SCRATCH_BYTES:
            raise ValueError(f"batch {B} needs {need} bytes of split-replay scratch; the static "
                             f"array holds {N.LS_SPLIT_STATIC_SCRATCH_BYTES}")
        with torch.cuda.device(self.device):  # the library checks that the pool's device is current
            rc = self.lib.ls_decode_step_split_static(self.handle, _ptr(slot_idx), B, _ptr(q),
                                                      _ptr(k), _ptr(v), _ptr(log_decay), _ptr(beta),
                                                      _ptr(y), C.c_void_p(_stream(stream)))
        N.check(rc, "ls_decode_step_split_static")
        return y

    def staging_bytes(self, batch: int) -> int:
        out = C.c_size_t(0)
        N.check(self.lib.ls_step_staging_bytes(self.handle, int(batch), C.byref(out)),
                "ls_step_staging_bytes")
        return int(out.value)

    def decode_step_host(self, slot_idx, q, k, v, log_decay, beta, y, stream=None):
        """ls_decode_step_host: host (pinned) inputs and output; the copies run
        inside the library on ``stream``.  Synchronize before reading y."""
        B = int(slot_idx.numel())
        cpu, f32 = torch.device("cpu"), torch.float32
        _need(slot_idx, "slot_idx", torch.int32, cpu, (B,))
        _need(q, "q", f32, cpu, (B, self.H, self.d_k))
        _need(k, "k", f32, cpu, (B, self.H, self.d_k))
        _need(v, "v", f32, cpu, (B, self.H, self.d_v))
        _need(log_decay, "log_decay", f32, cpu,
              (B, self.H) if self.dl == 1 else (B, self.H, self.d_k))
        _need(beta, "beta", f32, cpu, (B, self.H))
        _need(y, "y", f32, cpu, (B, self.H, self.d_v))
        need = self.staging_bytes(B)
        if self._staging is None or self._staging.numel() < need + 256:
            self._staging = torch.empty(need + 256, dtype=torch.uint8, device=self.device)
        sp = self._staging.data_ptr() + ((-self._staging.data_ptr()) % 256)
        rc = self.lib.ls_decode_step_host(self.handle, _ptr(slot_idx), B, _ptr(q), _ptr(k),
                                          _ptr(v), _ptr(log_decay), _ptr(beta), _ptr(y),
                                          C.c_void_p(sp), need, C.c_void_p(_stream(stream)))
        N.check(rc, "ls_decode_step_host")
        return y

    def window_commit(self, slots, stream=None):
        slots = self._slots(slots)
        N.check(self.lib.ls_window_commit(self.handle, _ptr(slots), int(slots.numel()),
                                          C.c_void_p(_stream(stream))), "ls_window_commit")

    def read(self, slots, out=None, stream=None) -> torch.Tensor:
        """Logical states [n, H, d_k, d_v] (FP32) of ``slots``."""
        slots = self._slots(slots)
        n = int(slots.numel())
        if out is None:
            out = torch.empty(n, self.H, self.d_k, self.d_v, dtype=torch.float32,
                              device=self.device)
        _need(out, "out", torch.float32, self.device, (n, self.H, self.d_k, self.d_v))
        N.check(self.lib.ls_pool_read(self.handle, _ptr(slots), n, _ptr(out),
                                      C.c_void_p(_stream(stream))), "ls_pool_read")
        return out

    def load(self, slots, state: torch.Tensor, stream=None):
        slots = self._slots(slots)
        n = int(slots.numel())
        _need(state, "state", torch.float32, self.device, (n, self.H, self.d_k, self.d_v))
        N.check(self.lib.ls_pool_load(self.handle, _ptr(slots), n, _ptr(state),
                                      C.c_void_p(_stream(stream))), "ls_pool_load")

    def reset(self, slots, stream=None):
        slots = self._slots(slots)
        N.check(self.lib.ls_pool_reset_slots(self.handle, _ptr(slots), int(slots.numel()),
                                             C.c_void_p(_stream(stream))), "ls_pool_reset_slots")

    def read_int8(self, slots, stream=None):
        """(codes [n, H, d_k, d_v] int8, key-row factors [n, H, d_k] float32) of
        the INT8 base: per-row scales, or the smoothing factors c (col_scales)."""
        slots = self._slots(slots)
        n = int(slots.numel())
        codes = torch.empty(n, self.H, self.d_k, self.d_v, dtype=torch.int8, device=self.device)
        scales = torch.empty(n, self.H, self.d_k, dtype=torch.float32, device=self.device)
        N.check(self.lib.ls_pool_read_int8(self.handle, _ptr(slots), n, _ptr(codes),
                                           _ptr(scales), C.c_void_p(_stream(stream))),
                "ls_pool_read_int8")
        return codes, scales

    def read_int8_col_scales(self, slots, stream=None):
        """col_scales pools: the per-value-column scales b [n, H, d_v] float32."""
        slots = self._slots(slots)
        n = int(slots.numel())
        b = torch.empty(n, self.H, self.d_v, dtype=torch.float32, device=self.device)
        N.check(self.lib.ls_pool_read_int8_col_scales(self.handle, _ptr(slots), n, _ptr(b),
                                                      C.c_void_p(_stream(stream))),
                "ls_pool_read_int8_col_scales")
        return b

    def read_compensators(self, slots, stream=None):
        """compensator pools: the current pairs (K~ [n, H, r, d_k], U~ [n, H, r, d_v])."""
        slots = self._slots(slots)
        n = int(slots.numel())
        r = self.compensators
        kk = torch.empty(n, self.H, r, self.d_k, dtype=torch.float32, device=self.device)
        uu = torch.empty(n, self.H, r, self.d_v, dtype=torch.float32, device=self.device)
        N.check(self.lib.ls_pool_read_compensators(self.handle, _ptr(slots), n, _ptr(kk), _ptr(uu),
                                                   C.c_void_p(_stream(stream))),
                "ls_pool_read_compensators")
        return kk, uu

    def read_log_meta(self, slots, stream=None):
        """(live log length [n, H] int32, cumulative log-decay [n, H, dl] float32)."""
        slots = self._slots(slots)
        n = int(slots.numel())
        ln = torch.empty(n, self.H, dtype=torch.int32, device=self.device)
        lb = torch.empty(n, self.H, self.dl, dtype=torch.float32, device=self.device)
        N.check(self.lib.ls_pool_read_log_meta(self.handle, _ptr(slots), n, _ptr(ln), _ptr(lb),
                                               C.c_void_p(_stream(stream))),
                "ls_pool_read_log_meta")
        return ln, lb

    def status(self, stream=None) -> int:
        """Synchronize, return and clear the device status word (LS_DEV_* bits)."""
        out = C.c_int32(0)
        N.check(self.lib.ls_pool_status(self.handle, C.c_void_p(_stream(stream)),
                                        C.byref(out)), "ls_pool_status")
        return int(out.value)
