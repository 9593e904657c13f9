"""Seeded synthetic workloads for the decode step.

This module is the one piece both the CUDA path's tests/benchmark and the CPU
oracle draw from: it produces the per-token inputs (q, k, v, log-decay,
beta) and the slot permutation of each workload.  It holds none of the
method's arithmetic (no state update, no quantization); it only samples the
input laws below.

Input laws (the pages measure on model activations and text corpora that are
not available here; these seeded laws stand in for their shapes -- d_k = d_v =
128, 32 heads as in the LeapQuant kernel study (§4.3) and the DeltaLog kernel
study (Table 3), 48 heads as in the STEPQuant reading notes):

* q, k ~ N(0, 1) per entry, then L2-normalised over d_k; v ~ N(0, 1);
  beta = sigmoid(N(0, 1)); the gate is given as the log-decay
  lambda = -softplus(N(0, 1)) * c (so alpha = exp(lambda) = exp(-softplus(x) c)).
* outlier key channels: a fixed Bernoulli(p) mask over (head, key channel)
  multiplies the raw key entry by a factor before normalisation.
* long-lived KDA channels: a fixed fraction of (head, key channel) pairs uses
  a much smaller multiplier c, so that their decay stays close to 1.
* heavy-tailed keys: raw key entries ~ Student-t(3) = N(0,1) / sqrt(chi2_3 / 3).

Each token's inputs come from a generator seeded with (workload seed, token
index), so any token can be regenerated on any device without the others.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

GATE_SCALAR = "scalar"    # Gated DeltaNet: one log-decay per head and token
GATE_PER_KEY = "per_key"  # KDA: one log-decay per key channel


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    gate: str
    batch: int            # B, requests decoded per token
    heads: int            # H
    d_k: int
    d_v: int
    tokens: int           # T
    pools: int            # independent layer pools
    num_slots: int        # P, slots in each pool
    windows: Sequence[int]  # INT8 windows W to exercise
    merge_interval: int   # deferred-log merge interval M
    seed: int
    lam_scale: float = 0.1
    k_law: str = "gauss"           # "gauss" or "student_t3"
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    longlived_frac: float = 0.0
    longlived_scale: float = 0.001
    permute_slots: bool = False
    prewarm_tokens: int = 0

    @property
    def dl(self) -> int:
        return 1 if self.gate == GATE_SCALAR else self.d_k

    @property
    def heads_per_pool(self) -> int:
        return self.batch * self.heads


# The five workloads, in order.  Readings where the description is open are
# stated in the design notes (window/merge choices for the drift workload, the
# shape of the outlier and long-lived masks, the pre-warm law).
WORKLOADS = [
    Workload("gdn_b1_h4_t64", GATE_SCALAR, batch=1, heads=4, d_k=128, d_v=128,
             tokens=64, pools=1, num_slots=1, windows=(16,), merge_interval=16,
             seed=0, lam_scale=0.1),
    Workload("gdn_pool_b64_h48_t1024_outliers", GATE_SCALAR, batch=64, heads=48,
             d_k=128, d_v=128, tokens=1024, pools=1, num_slots=64, windows=(64,),
             merge_interval=64, seed=1, lam_scale=0.1, outlier_frac=0.01,
             outlier_scale=20.0, permute_slots=True),
    Workload("kda_b128_h32_t512_longlived", GATE_PER_KEY, batch=128, heads=32,
             d_k=128, d_v=128, tokens=512, pools=1, num_slots=128, windows=(32,),
             merge_interval=16, seed=2, lam_scale=0.05, longlived_frac=0.10,
             longlived_scale=0.001),
    Workload("gdn_serving_b256_h48_4pools", GATE_SCALAR, batch=256, heads=48,
             d_k=128, d_v=128, tokens=128, pools=4, num_slots=256,
             windows=(8, 16, 32, 64, 128), merge_interval=16, seed=3,
             lam_scale=0.1, prewarm_tokens=256),
    Workload("kda_drift_b32_h32_t8192_studentt", GATE_PER_KEY, batch=32, heads=32,
             d_k=128, d_v=128, tokens=8192, pools=1, num_slots=32, windows=(32,),
             merge_interval=16, seed=4, lam_scale=0.05, k_law="student_t3",
             longlived_frac=0.10, longlived_scale=0.001),
]

WORKLOAD_BY_NAME = {w.name: w for w in WORKLOADS}


def custom(name="custom", gate=GATE_SCALAR, batch=2, heads=3, tokens=8, num_slots=None,
           windows=(4,), merge_interval=4, seed=123, **kw) -> Workload:
    """A small workload with the same input laws, for tests."""
    return Workload(name, gate, batch=batch, heads=heads, d_k=kw.pop("d_k", 128),
                    d_v=kw.pop("d_v", 128), tokens=tokens, pools=kw.pop("pools", 1),
                    num_slots=num_slots if num_slots is not None else batch,
                    windows=tuple(windows), merge_interval=merge_interval, seed=seed, **kw)


def _generator(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + int(stream) * 7_919 + 17) % (2 ** 63 - 1))
    return g


def _l2_normalise(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def static_masks(w: Workload, device="cpu"):
    """The fixed (head, key channel) masks of a workload: outliers, long-lived."""
    g = _generator(device, w.seed, 999_983)
    outl = torch.zeros(w.heads, w.d_k, dtype=torch.bool, device=device)
    longl = torch.zeros(w.heads, w.d_k, dtype=torch.bool, device=device)
    if w.outlier_frac > 0:
        outl = torch.rand(w.heads, w.d_k, generator=g, device=device) < w.outlier_frac
    if w.longlived_frac > 0:
        longl = torch.rand(w.heads, w.d_k, generator=g, device=device) < w.longlived_frac
    return outl, longl


def slot_index(w: Workload, device="cpu") -> torch.Tensor:
    """int32 [B]: the pool slot that batch row b decodes."""
    if w.permute_slots:
        g = _generator("cpu", w.seed, 999_979)
        perm = torch.randperm(w.num_slots, generator=g)[: w.batch]
    else:
        perm = torch.arange(w.batch)
    return perm.to(torch.int32).to(device)


def step_inputs(w: Workload, token: int, pool: int = 0, device="cpu",
                masks=None, rows: Optional[torch.Tensor] = None):
    """Inputs of one token for one pool.

    Returns float32 tensors q, k [B, H, d_k], v [B, H, d_v], lam [B, H] (scalar
    gate) or [B, H, d_k] (per-key gate), beta [B, H].  ``token`` may be negative
    for pre-warm tokens.  ``rows`` (optional) selects batch rows after sampling,
    so a subset is bit-identical to the same rows of the full draw.
    """
    if masks is None:
        masks = static_masks(w, device)
    outl, longl = masks
    B, H, dk, dv = w.batch, w.heads, w.d_k, w.d_v
    g = _generator(device, w.seed, (pool + 1) * 10_000_019 + token)
    f32 = torch.float32
    q = torch.randn(B, H, dk, generator=g, device=device, dtype=f32)
    kraw = torch.randn(B, H, dk, generator=g, device=device, dtype=f32)
    if w.k_law == "student_t3":
        chi = torch.randn(3, B, H, dk, generator=g, device=device, dtype=f32).pow(2).sum(0)
        kraw = kraw / torch.sqrt(chi / 3.0).clamp_min(1e-20)
    elif w.k_law != "gauss":
        raise ValueError(w.k_law)
    if w.outlier_frac > 0:
        kraw = torch.where(outl.unsqueeze(0), kraw * w.outlier_scale, kraw)
    v = torch.randn(B, H, dv, generator=g, device=device, dtype=f32)
    xb = torch.randn(B, H, generator=g, device=device, dtype=f32)
    if w.gate == GATE_SCALAR:
        xl = torch.randn(B, H, generator=g, device=device, dtype=f32)
        lam = -torch.nn.functional.softplus(xl) * w.lam_scale
    else:
        xl = torch.randn(B, H, dk, generator=g, device=device, dtype=f32)
        scale = torch.where(longl, torch.full_like(longl, w.longlived_scale, dtype=f32),
                            torch.full_like(longl, w.lam_scale, dtype=f32))
        lam = -torch.nn.functional.softplus(xl) * scale.unsqueeze(0)
    q = _l2_normalise(q)
    k = _l2_normalise(kraw)
    beta = torch.sigmoid(xb)
    out = [q, k, v, lam.contiguous(), beta]
    if rows is not None:
        out = [t[rows] for t in out]
    return tuple(t.contiguous() for t in out)


def initial_state(w: Workload, device="cpu", scale: float = 1.0) -> torch.Tensor:
    """A seeded dense start state [P, H, d_k, d_v] with N(0, scale^2) entries
    (used by tests that start windows from a non-zero state)."""
    g = _generator(device, w.seed, 999_961)
    return torch.randn(w.num_slots, w.heads, w.d_k, w.d_v, generator=g, device=device,
                       dtype=torch.float32) * scale
