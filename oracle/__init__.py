"""Double-precision CPU oracle for the recurrent-state decode step.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package; the product path (the
CUDA library ``libls`` and its binding) never does.  It shares no code with the
CUDA path: the arithmetic lives in ``ls_oracle.c``; this module only holds the
numpy arrays of each state and marshals them through ctypes.

Each class keeps ``nstates`` independent head states, addressed by an index
array: row ``r`` of a batch updates state ``idx[r]``.  Inputs are float32
arrays shaped ``[n, d]`` (``lam`` is ``[n, 1]`` for the scalar gate of Gated
DeltaNet, ``[n, d_k]`` for the per-key gate of KDA; ``beta`` is ``[n]``).
States are returned in the logical layout ``[.., d_k, d_v]``.

Page references: "LeapQuant: Efficient Linear Attention with Accurate Recurrent
State Quantization" (eager form App. A, per-window scheme §3.2 eq. 3-4, eq. 9,
App. B.3) and "DeltaLog: Deferred Materialization of Recurrent States for
Linear Attention Decoding" (§3.1 Algorithm 1, eq. 4-7).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import LIB, build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = C.CDLL(LIB)
        P = C.c_void_p
        I64, I32 = C.c_int64, C.c_int
        lib.orc_max_threads.restype = I32
        lib.orc_eager_step.argtypes = [I64, I32, I32, I32, I32, P, P, P, P, P, P, P, P, I32]
        lib.orc_deferred_step.argtypes = [I64, I32, I32, I32, I32, I32, I32, P, P, P, P, P, P,
                                          P, P, P, P, P, P, P, I32]
        lib.orc_deferred_logical.argtypes = [I64, I32, I32, I32, I32, P, P, P, P, P, P, P, P]
        lib.orc_deferred_commit.argtypes = [I64, I32, I32, I32, I32, P, P, P, P, P, P, P]
        lib.orc_quantize_rows.argtypes = [I64, I32, I32, P, P, P]
        lib.orc_dequantize_rows.argtypes = [I64, I32, I32, P, P, P]
        lib.orc_quantize_cols.argtypes = [I64, I32, I32, P, P, P, P]
        lib.orc_fit_compensators.argtypes = [I64, I32, I32, I32, P, P, P, I32]
        lib.orc_dequantize_cols.argtypes = [I64, I32, I32, P, P, P, P]
        lib.orc_window_step.argtypes = [I64, I32, I32, I32, I32, I32, I32, I32, P, P, P, P, P,
                                        P, P, P, P, P, P, P, P, P, P, P, P, I32]
        lib.orc_window_commit.argtypes = [I64, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P]
        lib.orc_window_load.argtypes = [I64, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P]
        lib.orc_window_unrolled.argtypes = [I64, I32, I32, I32, I32, I32, I32, P, P, P, P, P,
                                            P, P, P, P, P, P]
        lib.orc_window_readout.argtypes = [I64, I32, I32, I32, I32, I32, I32, P, P, P, P, P,
                                           P, P, P, P, P, P, P]
        for name in ("orc_eager_step", "orc_deferred_step", "orc_deferred_logical",
                     "orc_deferred_commit", "orc_quantize_rows", "orc_dequantize_rows",
                     "orc_quantize_cols", "orc_dequantize_cols", "orc_fit_compensators",
                     "orc_window_step", "orc_window_commit", "orc_window_load",
                     "orc_window_unrolled", "orc_window_readout"):
            getattr(lib, name).restype = I32
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().orc_max_threads())


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _f32(a, shape=None) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if shape is not None:
        a = a.reshape(shape)
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


class _Base:
    def __init__(self, nstates: int, dk: int, dv: int, dl: int, nthreads: int = 0):
        if dl not in (1, dk):
            raise ValueError("dl must be 1 (scalar gate) or d_k (per-key gate)")
        self.n, self.dk, self.dv, self.dl = int(nstates), int(dk), int(dv), int(dl)
        self.nthreads = int(nthreads)

    def _idx(self, idx) -> np.ndarray:
        idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1))
        if idx.size and (idx.min() < 0 or idx.max() >= self.n):
            raise IndexError("state index out of range")
        if np.unique(idx).size != idx.size:
            raise ValueError("rows must name distinct states")
        return idx

    def _inputs(self, idx, q, k, v, lam, beta):
        n = idx.size
        return (_f32(q, (n, self.dk)), _f32(k, (n, self.dk)), _f32(v, (n, self.dv)),
                _f32(lam, (n, self.dl)), _f32(beta, (n,)))


class EagerOracle(_Base):
    """Eager recurrence of every state (LeapQuant App. A with eq. 1).

    plain=True: the update pair (k, v) without the delta-rule correction
    (DeltaLog Table 1, the linear attention / RetNet / GLA / RWKV6 rows)."""

    def __init__(self, nstates, dk, dv, dl, nthreads=0, plain=False):
        super().__init__(nstates, dk, dv, dl, nthreads)
        self.rule = 1 if plain else 0
        self.S = np.zeros((self.n, dk, dv), dtype=np.float64)

    def step(self, idx, q, k, v, lam, beta) -> np.ndarray:
        idx = self._idx(idx)
        q, k, v, lam, beta = self._inputs(idx, q, k, v, lam, beta)
        y = np.zeros((idx.size, self.dv), dtype=np.float64)
        _check(_load().orc_eager_step(idx.size, self.rule, self.dk, self.dv, self.dl, _p(self.S),
                                      _p(idx),
                                      _p(q), _p(k), _p(v), _p(lam), _p(beta), _p(y),
                                      self.nthreads), "eager step")
        return y

    def logical(self, idx) -> np.ndarray:
        return self.S[self._idx(idx)].copy()

    def load(self, idx, S):
        self.S[self._idx(idx)] = np.asarray(S, dtype=np.float64)

    def reset(self, idx):
        self.S[self._idx(idx)] = 0.0

    def commit(self, idx):
        self._idx(idx)


class DeferredOracle(_Base):
    """Base + bounded log, DeltaLog Algorithm 1 with merge interval M
    (plain=True: update pair (k, v), as EagerOracle; k16=True: key-side
    factors stored as bfloat16, DeltaLog §3.4)."""

    def __init__(self, nstates, dk, dv, dl, M, nthreads=0, plain=False, k16=False):
        super().__init__(nstates, dk, dv, dl, nthreads)
        if M < 1:
            raise ValueError("M >= 1")
        self.M = int(M)
        self.rule = 1 if plain else 0
        self.k16 = 1 if k16 else 0
        Cap = max(self.M - 1, 0)
        self.base = np.zeros((self.n, dk, dv), dtype=np.float64)
        self.lbar = np.zeros((self.n, dl), dtype=np.float64)
        # one spare entry so that the arrays are never empty (M = 1)
        self.K = np.zeros((self.n, max(Cap, 1), dk), dtype=np.float64)
        self.U = np.zeros((self.n, max(Cap, 1), dv), dtype=np.float64)
        self.Lam = np.zeros((self.n, max(Cap, 1), dl), dtype=np.float64)
        self.L = np.zeros((self.n,), dtype=np.int32)
        if Cap == 0:
            # the C side indexes entries with stride C = M - 1 = 0
            pass

    def _arrays(self):
        return (_p(self.base), _p(self.lbar), _p(self.K), _p(self.U), _p(self.Lam), _p(self.L))

    def step(self, idx, q, k, v, lam, beta) -> np.ndarray:
        idx = self._idx(idx)
        q, k, v, lam, beta = self._inputs(idx, q, k, v, lam, beta)
        y = np.zeros((idx.size, self.dv), dtype=np.float64)
        self._stride_guard()
        _check(_load().orc_deferred_step(idx.size, self.rule, self.k16, self.dk, self.dv, self.dl,
                                         self.M,
                                         *self._arrays(), _p(idx), _p(q), _p(k), _p(v),
                                         _p(lam), _p(beta), _p(y), self.nthreads),
               "deferred step")
        return y

    def _stride_guard(self):
        # The C code addresses entries of state s at s*C*d; keep the numpy
        # arrays shaped [n, C, d] exactly (C >= 1) or [n, 1, d] when C == 0.
        Cap = self.M - 1
        assert self.K.shape[1] == max(Cap, 1)

    def logical(self, idx) -> np.ndarray:
        idx = self._idx(idx)
        out = np.zeros((idx.size, self.dk, self.dv), dtype=np.float64)
        _check(_load().orc_deferred_logical(idx.size, self.dk, self.dv, self.dl, self.M,
                                            *self._arrays(), _p(idx), _p(out)),
               "deferred logical")
        return out

    def commit(self, idx):
        idx = self._idx(idx)
        _check(_load().orc_deferred_commit(idx.size, self.dk, self.dv, self.dl, self.M,
                                           *self._arrays(), _p(idx)), "deferred commit")

    def load(self, idx, S):
        idx = self._idx(idx)
        self.base[idx] = np.asarray(S, dtype=np.float64)
        self.lbar[idx] = 0.0
        self.L[idx] = 0

    def reset(self, idx):
        self.load(idx, np.zeros((len(idx), self.dk, self.dv)))


class WindowInt8Oracle(_Base):
    """Per-window INT8 scheme, LeapQuant §3.2 eq. 3-4, window W.

    col_scales=False: one FP32 scale per key row.  col_scales=True: the
    smoothed per-value-column format of LeapQuant §3.4 eq. 7 / App. B.3
    (row factors = smoothing vector c, column factors = scales b).
    compensators=r: r Compensator Tokens (LeapQuant §3.3) fitted at every
    boundary; the residual is what is quantized.
    k16: bfloat16 keys in the records (DeltaLog §3.4).  r16: FP16 records,
    keys and values, and FP16 compensator pairs (LeapQuant §4.3)."""

    def __init__(self, nstates, dk, dv, dl, W, nthreads=0, col_scales=False, compensators=0,
                 k16=False, r16=False):
        super().__init__(nstates, dk, dv, dl, nthreads)
        if W < 1:
            raise ValueError("W >= 1")
        self.W = int(W)
        self.mode = 1 if col_scales else 0
        self.r = int(compensators)
        if k16 and r16:
            raise ValueError("k16 and r16 are exclusive")
        self.rec = 2 if r16 else (1 if k16 else 0)
        self.ck = np.zeros((self.n, max(self.r, 1), dk), dtype=np.float64)
        self.cu = np.zeros((self.n, max(self.r, 1), dv), dtype=np.float64)
        self.Z = np.zeros((self.n, dk, dv), dtype=np.int8)
        self.s = np.zeros((self.n, dk), dtype=np.float32)
        self.fc = np.zeros((self.n, dv), dtype=np.float32)
        self.Sw = np.zeros((self.n, dk, dv), dtype=np.float64)
        self.rl = np.zeros((self.n, self.W, dl), dtype=np.float64)
        self.rk = np.zeros((self.n, self.W, dk), dtype=np.float64)
        self.ru = np.zeros((self.n, self.W, dv), dtype=np.float64)
        self.cnt = np.zeros((self.n,), dtype=np.int32)

    def step(self, idx, q, k, v, lam, beta) -> np.ndarray:
        idx = self._idx(idx)
        q, k, v, lam, beta = self._inputs(idx, q, k, v, lam, beta)
        y = np.zeros((idx.size, self.dv), dtype=np.float64)
        _check(_load().orc_window_step(idx.size, self.mode, self.r, self.rec, self.dk, self.dv,
                                       self.dl,
                                       self.W, _p(self.Z), _p(self.s), _p(self.fc),
                                       _p(self.ck), _p(self.cu), _p(self.Sw),
                                       _p(self.rl),
                                       _p(self.rk), _p(self.ru), _p(self.cnt), _p(idx),
                                       _p(q), _p(k), _p(v), _p(lam), _p(beta), _p(y),
                                       self.nthreads), "window step")
        return y

    def logical(self, idx) -> np.ndarray:
        """The exact in-window state S_i (eq. 3), i.e. the logical state."""
        return self.Sw[self._idx(idx)].copy()

    def codes(self, idx):
        """(Z, row factors): per-key-row scales, or the smoothing vector c."""
        idx = self._idx(idx)
        return self.Z[idx].copy(), self.s[idx].copy()

    def col_factors(self, idx):
        """The per-value-column scales b (smoothed format; zeros otherwise)."""
        return self.fc[self._idx(idx)].copy()

    def compensators(self, idx):
        """The current window's compensator pairs (K~ [n, r, dk], U~ [n, r, dv])."""
        idx = self._idx(idx)
        return self.ck[idx, :self.r].copy(), self.cu[idx, :self.r].copy()

    def commit(self, idx):
        idx = self._idx(idx)
        _check(_load().orc_window_commit(idx.size, self.mode, self.r, self.rec, self.dk, self.dv,
                                         _p(self.Z), _p(self.s), _p(self.fc), _p(self.ck),
                                         _p(self.cu), _p(self.Sw), _p(self.cnt), _p(idx)),
               "window commit")

    def load(self, idx, S):
        idx = self._idx(idx)
        S = np.ascontiguousarray(np.asarray(S, dtype=np.float64).reshape(idx.size, self.dk,
                                                                          self.dv))
        _check(_load().orc_window_load(idx.size, self.mode, self.r, self.rec, self.dk, self.dv,
                                       _p(S),
                                       _p(self.Z), _p(self.s), _p(self.fc), _p(self.ck),
                                       _p(self.cu), _p(self.Sw), _p(self.cnt), _p(idx)),
               "window load")

    def reset(self, idx):
        self.load(idx, np.zeros((len(idx), self.dk, self.dv)))

    def unrolled(self, idx) -> np.ndarray:
        """S_l rebuilt from the boundary state and the buffered records (eq. 4)."""
        idx = self._idx(idx)
        out = np.zeros((idx.size, self.dk, self.dv), dtype=np.float64)
        _check(_load().orc_window_unrolled(idx.size, self.mode, self.r, self.dk, self.dv,
                                           self.dl, self.W, _p(self.Z), _p(self.s), _p(self.fc),
                                           _p(self.ck), _p(self.cu), _p(self.rl), _p(self.rk),
                                           _p(self.ru), _p(self.cnt), _p(idx), _p(out)),
               "window unrolled")
        return out

    def readout(self, idx, x) -> np.ndarray:
        """S_l^T x from the boundary state and the records, without S_l (eq. 9)."""
        idx = self._idx(idx)
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64).reshape(idx.size, self.dk))
        out = np.zeros((idx.size, self.dv), dtype=np.float64)
        _check(_load().orc_window_readout(idx.size, self.mode, self.r, self.dk, self.dv,
                                          self.dl, self.W, _p(self.Z), _p(self.s), _p(self.fc),
                                          _p(self.ck), _p(self.cu), _p(self.rl), _p(self.rk),
                                          _p(self.ru), _p(self.cnt), _p(idx), _p(x), _p(out)),
               "window readout")
        return out


def quantize_rows(S):
    """Symmetric INT8 with one FP32 scale per key row: returns (Z, s)."""
    S = np.ascontiguousarray(np.asarray(S, dtype=np.float64))
    lead = S.shape[:-2]
    dk, dv = S.shape[-2:]
    n = int(np.prod(lead)) if lead else 1
    Z = np.zeros(S.shape, dtype=np.int8)
    s = np.zeros(lead + (dk,), dtype=np.float32)
    _check(_load().orc_quantize_rows(n, dk, dv, _p(S), _p(Z), _p(s)), "quantize")
    return Z, s


def dequantize_rows(Z, s):
    Z = np.ascontiguousarray(np.asarray(Z, dtype=np.int8))
    s = np.ascontiguousarray(np.asarray(s, dtype=np.float32))
    lead = Z.shape[:-2]
    dk, dv = Z.shape[-2:]
    n = int(np.prod(lead)) if lead else 1
    S = np.zeros(Z.shape, dtype=np.float64)
    _check(_load().orc_dequantize_rows(n, dk, dv, _p(Z), _p(s), _p(S)), "dequantize")
    return S


def quantize_cols(S):
    """Smoothed per-value-column INT8 (LeapQuant §3.4 eq. 7, App. B.3):
    returns (Z, c, b) with S ~ c_i Z_ij b_j."""
    S = np.ascontiguousarray(np.asarray(S, dtype=np.float64))
    lead = S.shape[:-2]
    dk, dv = S.shape[-2:]
    n = int(np.prod(lead)) if lead else 1
    Z = np.zeros(S.shape, dtype=np.int8)
    c = np.zeros(lead + (dk,), dtype=np.float32)
    b = np.zeros(lead + (dv,), dtype=np.float32)
    _check(_load().orc_quantize_cols(n, dk, dv, _p(S), _p(Z), _p(c), _p(b)), "quantize cols")
    return Z, c, b


def dequantize_cols(Z, c, b):
    Z = np.ascontiguousarray(np.asarray(Z, dtype=np.int8))
    c = np.ascontiguousarray(np.asarray(c, dtype=np.float32))
    b = np.ascontiguousarray(np.asarray(b, dtype=np.float32))
    lead = Z.shape[:-2]
    dk, dv = Z.shape[-2:]
    n = int(np.prod(lead)) if lead else 1
    S = np.zeros(Z.shape, dtype=np.float64)
    _check(_load().orc_dequantize_cols(n, dk, dv, _p(Z), _p(c), _p(b), _p(S)), "dequantize cols")
    return S


def fit_compensators(S, r, warm_cu=None):
    """LeapQuant §3.3 Compensator Tokens fitted to S [..., dk, dv] by the
    oracle's power iteration: returns (residual, K~ [..., r, dk], U~ [..., r, dv])."""
    S = np.array(S, dtype=np.float64, copy=True, order="C")
    lead = S.shape[:-2]
    dk, dv = S.shape[-2:]
    n = int(np.prod(lead)) if lead else 1
    ck = np.zeros(lead + (r, dk), dtype=np.float64)
    cu = np.zeros(lead + (r, dv), dtype=np.float64)
    if warm_cu is not None:
        cu[...] = warm_cu
    _check(_load().orc_fit_compensators(n, int(r), dk, dv, _p(S), _p(ck), _p(cu),
                                        1 if warm_cu is not None else 0), "fit compensators")
    return S, ck, cu


__all__ = ["EagerOracle", "DeferredOracle", "WindowInt8Oracle", "quantize_rows",
           "dequantize_rows", "quantize_cols", "dequantize_cols", "fit_compensators",
           "max_threads", "build_oracle"]
