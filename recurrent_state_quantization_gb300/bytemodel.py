"""Algorithmic HBM bytes of one decode step, per (request, head).

These are the bytes the method has to move, independent of how a kernel is
written; the roofline fraction divides them by a measured kernel time.

* Token inputs and output, every variant: q, k, v read and y written (4 d
  bytes each), beta (4 B), log-decay (4 dl B, dl = 1 scalar gate / d_k per-key
  gate), slot index (4 B).
* Eager FP32: read and write the dense state, 2 * 4 d_k d_v ("DeltaLog:
  Deferred Materialization of Recurrent States for Linear Attention
  Decoding", §3.2 eq. 8: T_dense = T_common + 2 C_state).
* Deferred base + log with merge interval M (DeltaLog §3.2 eq. 9-11):
  C_state (base read every token) + C_state / M (one base write per cycle)
  + C_log(M) = ((M-1)/M + (M-1)/2) C_entry (appends + replay reads) + 2 C_decay,
  with C_entry = p_K d_k + p_U d_v + 4 dl and C_decay = 4 dl.
* Per-window INT8 with window W ("LeapQuant: Efficient Linear Attention with
  Accurate Recurrent State Quantization", §3.2): the same cycle with an INT8
  base plus one FP32 scale per key row in place of the FP32 base; the
  smoothed per-value-column format (§3.4 eq. 7, App. B.3) adds one FP32
  scale per value column to that base; r Compensator Tokens (§3.3) add r
  log entries read by every token and written once per window.
* bfloat16 key-side log factors (DeltaLog §3.4): p_K = 2 in C_entry.
* FP16 records (LeapQuant §4.1, §4.3): p_K = p_U = 2 in C_entry, for the
  window's records and the compensator pairs alike.
"""
from __future__ import annotations

GIB = 1024.0 ** 3


def _dl(gate: str, d_k: int) -> int:
    return 1 if gate == "scalar" else d_k


def io_bytes(gate: str, d_k: int = 128, d_v: int = 128) -> int:
    return 4 * (2 * d_k + 2 * d_v) + 4 + 4 * _dl(gate, d_k) + 4


def entry_bytes(gate: str, d_k: int = 128, d_v: int = 128, p_k: int = 4, p_u: int = 4) -> int:
    return p_k * d_k + p_u * d_v + 4 * _dl(gate, d_k)


def state_bytes_fp32(d_k: int = 128, d_v: int = 128) -> int:
    return 4 * d_k * d_v


def state_bytes_int8(d_k: int = 128, d_v: int = 128, col_scales: bool = False) -> int:
    return d_k * d_v + 4 * d_k + (4 * d_v if col_scales else 0)


def eager_bytes(gate: str, d_k: int = 128, d_v: int = 128) -> float:
    return 2 * state_bytes_fp32(d_k, d_v) + io_bytes(gate, d_k, d_v)


def log_cycle_bytes(base: float, gate: str, M: int, d_k: int = 128, d_v: int = 128,
                    p_k: int = 4, p_u: int = 4) -> float:
    e = entry_bytes(gate, d_k, d_v, p_k, p_u)
    c_log = ((M - 1) / M + (M - 1) / 2) * e
    return base * (1 + 1 / M) + c_log + 2 * 4 * _dl(gate, d_k) + io_bytes(gate, d_k, d_v)


def deferred_bytes(gate: str, M: int, d_k: int = 128, d_v: int = 128, p_k: int = 4) -> float:
    return log_cycle_bytes(state_bytes_fp32(d_k, d_v), gate, M, d_k, d_v, p_k)


def int8_bytes(gate: str, W: int, d_k: int = 128, d_v: int = 128, col_scales: bool = False,
               compensators: int = 0, p_k: int = 4, p_u: int = 4) -> float:
    comp = compensators * entry_bytes(gate, d_k, d_v, p_k, p_u) * (1 + 1 / W)
    return log_cycle_bytes(state_bytes_int8(d_k, d_v, col_scales), gate, W, d_k, d_v,
                           p_k, p_u) + comp


def variant_bytes(variant: str, gate: str, window: int = 1) -> float:
    if variant == "eager":
        return eager_bytes(gate)
    if variant == "deferred":
        return deferred_bytes(gate, window)
    if variant == "int8":
        return int8_bytes(gate, window)
    raise ValueError(variant)


def flops_per_head_step(d_k: int = 128, d_v: int = 128, live_log: float = 0.0) -> float:
    """Two GEMVs and a rank-1 update (6 d_k d_v) plus 4 L d replay FLOPs."""
    return 6 * d_k * d_v + 4 * live_log * (d_k + d_v) / 2


def leapquant_boundary_bytes_per_elem(d_k: int = 128, d_v: int = 128, r: int = 4,
                                      value_scales: bool = True, smoothing: bool = True) -> float:
    """Bytes per state element of a LeapQuant window-boundary state: INT8
    residual, FP32 per-value-channel scales (App. B.3), FP32 key-row smoothing
    scales (§3.4) and r FP16 compensator pairs (§3.3)."""
    b = d_k * d_v + (4 * d_v if value_scales else 0) + (4 * d_k if smoothing else 0)
    b += r * (d_k + d_v) * 2
    return b / (d_k * d_v)


def leapquant_record_buffer_bytes(p: int, gate: str = "scalar", d_k: int = 128, d_v: int = 128,
                                  bytes_per_value: int = 2) -> int:
    """Per-head buffer of p records (alpha, k, u) (LeapQuant §3.2, §4.3)."""
    return p * (_dl(gate, d_k) + d_k + d_v) * bytes_per_value
