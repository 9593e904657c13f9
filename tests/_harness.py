"""Helpers shared by the GPU parity tests: drive a StatePool and the CPU
oracle with the same seeded inputs and compare.  Test infrastructure only."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from recurrent_state_quantization_gb300 import StatePool
from recurrent_state_quantization_gb300 import workloads as wl

D = 128


def make_oracle(variant, nstates, dl, window, nthreads=0, col_scales=False, compensators=0,
                plain=False, k16=False, r16=False):
    if variant == "eager":
        return oracle.EagerOracle(nstates, D, D, dl, nthreads, plain=plain)
    if variant == "deferred":
        return oracle.DeferredOracle(nstates, D, D, dl, window, nthreads, plain=plain, k16=k16)
    if variant == "int8":
        return oracle.WindowInt8Oracle(nstates, D, D, dl, window, nthreads, col_scales=col_scales,
                                       compensators=compensators, k16=k16, r16=r16)
    raise ValueError(variant)


def relmax(a, b):
    """Max |a - b| / max |b| (per tensor)."""
    den = float(np.abs(b).max())
    return float(np.abs(a - b).max()) / (den if den > 0 else 1.0)


def rel_l2(a, b):
    den = float(np.linalg.norm(b))
    return float(np.linalg.norm(a - b)) / (den if den > 0 else 1.0)


@dataclasses.dataclass
class Sample:
    """Batch rows (b, h) followed on the oracle side."""
    rows: np.ndarray       # flat row indices b*H + h into the [B*H] step arrays
    state_idx: np.ndarray  # oracle state index slot*H + h of each row


def sample_rows(w: wl.Workload, slot_idx: torch.Tensor, n=None, seed=0) -> Sample:
    B, H = w.batch, w.heads
    all_rows = np.arange(B * H)
    if n is not None and n < B * H:
        rng = np.random.default_rng(seed)
        rows = np.sort(rng.choice(B * H, n, replace=False))
    else:
        rows = all_rows
    slots = slot_idx.cpu().numpy().astype(np.int64)
    state = slots[rows // H] * H + rows % H
    return Sample(rows=rows, state_idx=state)


def host_inputs(inputs, w: wl.Workload, rows: np.ndarray):
    q, k, v, lam, beta = inputs
    n = w.batch * w.heads
    rr = torch.as_tensor(rows, device=q.device)
    f = lambda t, d: t.reshape(n, d).index_select(0, rr).cpu().numpy()
    return (f(q, D), f(k, D), f(v, D), f(lam, w.dl), beta.reshape(n).index_select(0, rr)
            .cpu().numpy())


class Pair:
    """A GPU pool and an oracle stepped together over a workload."""

    def __init__(self, w: wl.Workload, variant: str, window: int, n_sample=None, device="cuda",
                 seed=0, nthreads=0, col_scales=False, compensators=0, plain=False, k16=False,
                 split=False, r16=False):
        self.w, self.variant, self.window = w, variant, window
        self.split = bool(split)  # drive the pool through the split-replay entry point
        self.col_scales = bool(col_scales)
        self.compensators = int(compensators)
        self.r16 = bool(r16)
        self.dev = torch.device(device)
        self.pool = StatePool(w.num_slots, w.heads, variant, w.gate, window, device=self.dev,
                              col_scales=col_scales, compensators=compensators, plain=plain,
                              k16=k16, r16=r16)
        self.orc = make_oracle(variant, w.num_slots * w.heads, w.dl, window, nthreads,
                               col_scales=col_scales, compensators=compensators, plain=plain,
                               k16=k16, r16=r16)
        self.slot_idx = wl.slot_index(w, self.dev)
        self.sample = sample_rows(w, self.slot_idx, n_sample, seed)
        self.masks = wl.static_masks(w, self.dev)
        self.worst_y = 0.0
        self.worst_y_l2 = 0.0
        self._y_num = {}
        self._y_den = {}

    def step(self, t: int, pool_id: int = 0, slot_idx=None, rows=None):
        w = self.w
        inputs = wl.step_inputs(w, t, pool=pool_id, device=self.dev, masks=self.masks)
        if self.split:
            y = self.pool.decode_step_split(self.slot_idx, *inputs)
        else:
            y = self.pool.decode_step(self.slot_idx, *inputs)
        s = self.sample
        hq = host_inputs(inputs, w, s.rows)
        yo = self.orc.step(s.state_idx, *hq)
        yg = y.reshape(-1, D).index_select(0, torch.as_tensor(s.rows, device=self.dev))
        yg = yg.double().cpu().numpy()
        # per (head) max error over the run, normalised by the head's largest |y|
        for r, (a, b) in enumerate(zip(yg, yo)):
            self._y_num[r] = max(self._y_num.get(r, 0.0), float(np.abs(a - b).max()))
            self._y_den[r] = max(self._y_den.get(r, 0.0), float(np.abs(b).max()))
            self._l2n = getattr(self, "_l2n", {})
            self._l2d = getattr(self, "_l2d", {})
            self._l2n[r] = self._l2n.get(r, 0.0) + float(((a - b) ** 2).sum())
            self._l2d[r] = self._l2d.get(r, 0.0) + float((b ** 2).sum())
        return y, yo

    def force_boundary(self):
        """Restart every sampled state from the oracle's own current state.

        The oracle's logical state (at a window boundary) is rounded to FP32
        and that one array is loaded into both the oracle and the GPU pool, so
        the next window starts from identical boundary codes on both sides.
        Only oracle values flow, into both sides; no GPU value reaches the
        oracle.  Heads of the touched slots that are not sampled keep the GPU's
        own state (read, then loaded back).
        """
        w, s = self.w, self.sample
        S32 = self.orc.logical(s.state_idx).astype(np.float32)
        slots_b = self.slot_idx.cpu().numpy()[s.rows // w.heads]
        uniq = np.unique(slots_b)
        ut = torch.as_tensor(uniq, dtype=torch.int32, device=self.dev)
        cur = self.pool.read(ut).cpu()
        pos = {int(x): i for i, x in enumerate(uniq)}
        for n_, r in enumerate(s.rows):
            cur[pos[int(slots_b[n_])], r % w.heads] = torch.from_numpy(S32[n_])
        self.pool.load(ut, cur.to(self.dev))
        self.orc.load(s.state_idx, S32.astype(np.float64))

    def y_err(self) -> float:
        return max((self._y_num[r] / self._y_den[r] if self._y_den[r] > 0 else self._y_num[r])
                   for r in self._y_num)

    def y_rel_l2(self) -> float:
        return max(np.sqrt(self._l2n[r] / self._l2d[r]) if self._l2d[r] > 0 else 0.0
                   for r in self._l2n)

    def state_err(self) -> float:
        """Max over sampled heads of max|S_gpu - S_orc| / max|S_orc| (logical states)."""
        w, s = self.w, self.sample
        slots_b = self.slot_idx.cpu().numpy()[s.rows // w.heads]
        uniq = np.unique(slots_b)
        S = self.pool.read(torch.as_tensor(uniq, dtype=torch.int32)).double().cpu().numpy()
        pos = {int(x): i for i, x in enumerate(uniq)}
        worst = 0.0
        So = self.orc.logical(s.state_idx)
        for n_, r in enumerate(s.rows):
            g = S[pos[int(slots_b[n_])], r % w.heads]
            worst = max(worst, relmax(g, So[n_]))
        return worst

    def factor_err(self):
        """INT8: max relative error of the key-row factors (scales or smoothing
        factors c) and, for the column format, of the column scales b, over
        the sampled heads."""
        w, s = self.w, self.sample
        slots_b = self.slot_idx.cpu().numpy()[s.rows // w.heads]
        uniq = np.unique(slots_b)
        ut = torch.as_tensor(uniq, dtype=torch.int32, device=self.dev)
        _, fr = self.pool.read_int8(ut)
        fr = fr.cpu().numpy()
        fc = self.pool.read_int8_col_scales(ut).cpu().numpy() if self.col_scales else None
        pos = {int(x): i for i, x in enumerate(uniq)}
        _, fro = self.orc.codes(s.state_idx)
        fco = self.orc.col_factors(s.state_idx)
        mag = np.abs(self.orc.logical(s.state_idx)).reshape(len(s.rows), -1).max(axis=1)
        worst = 0.0
        for n_, r in enumerate(s.rows):
            o_r = fro[n_].astype(np.float64)
            o_c = fco[n_].astype(np.float64) if fc is not None else np.ones(1)
            # compensator pools: factors of residual rows / columns at the
            # rounding floor (see code_mismatch) are not determined
            keep_r = np.ones(o_r.shape, bool)
            keep_c = np.ones(o_c.shape, bool)
            if self.compensators:
                floor = (2.0 ** -18) * mag[n_] / 127.0
                keep_r = o_r * np.abs(o_c).max() > floor
                keep_c = np.abs(o_r).max() * o_c > floor
            g = fr[pos[int(slots_b[n_])], r % w.heads].astype(np.float64)
            rel = np.abs(g - o_r) / np.maximum(np.abs(o_r), 1e-30)
            worst = max(worst, float(np.max(rel[keep_r], initial=0.0)))
            if fc is not None:
                g = fc[pos[int(slots_b[n_])], r % w.heads].astype(np.float64)
                rel = np.abs(g - o_c) / np.maximum(np.abs(o_c), 1e-30)
                worst = max(worst, float(np.max(rel[keep_c], initial=0.0)))
        return worst

    def comp_err(self):
        """Compensator pools: max relative error of K~ U~^T (the pairs'
        contribution) over the sampled heads, against the oracle's."""
        w, s = self.w, self.sample
        slots_b = self.slot_idx.cpu().numpy()[s.rows // w.heads]
        uniq = np.unique(slots_b)
        kk, uu = self.pool.read_compensators(torch.as_tensor(uniq, dtype=torch.int32, device=self.dev))
        kk, uu = kk.double().cpu().numpy(), uu.double().cpu().numpy()
        pos = {int(x): i for i, x in enumerate(uniq)}
        ko, uo = self.orc.compensators(s.state_idx)
        worst = 0.0
        for n_, r in enumerate(s.rows):
            g = np.einsum("hi,hj->ij", kk[pos[int(slots_b[n_])], r % w.heads], uu[pos[int(slots_b[n_])], r % w.heads])
            o = np.einsum("hi,hj->ij", ko[n_], uo[n_])
            worst = max(worst, relmax(g, o))
        return worst

    def boundary_step_err(self):
        """INT8 at a window boundary: max over the sampled heads' elements of
        |S_gpu - S_orc| / (step_gpu / 2 + step_orc / 2 + 2^-10 max|S_orc|),
        S the logical (dequantized) states and step the code step of each
        side's own format (s_i, or c_i b_j with column scales).  Each side's
        boundary state lies within half its own step of its unquantized
        state, and the two unquantized states differ by FP32 rounding and by
        binary16 rounding flips of single record elements (2^-11 of a record,
        at most 2^-10 of the state), so the ratio is at most 1 whatever pairs
        each side fitted."""
        w, s = self.w, self.sample
        slots_b = self.slot_idx.cpu().numpy()[s.rows // w.heads]
        uniq = np.unique(slots_b)
        ut = torch.as_tensor(uniq, dtype=torch.int32, device=self.dev)
        S = self.pool.read(ut).double().cpu().numpy()
        _, fr = self.pool.read_int8(ut)
        fr = fr.double().cpu().numpy()
        fc = self.pool.read_int8_col_scales(ut).double().cpu().numpy() if self.col_scales else None
        pos = {int(x): i for i, x in enumerate(uniq)}
        So = self.orc.logical(s.state_idx)
        _, fro = self.orc.codes(s.state_idx)
        fco = self.orc.col_factors(s.state_idx) if self.col_scales else None
        worst = 0.0
        for n_, r in enumerate(s.rows):
            i = pos[int(slots_b[n_])]
            sg = fr[i, r % w.heads][:, None] * (fc[i, r % w.heads][None, :] if fc is not None else 1.0)
            so = fro[n_].astype(np.float64)[:, None] * (
                fco[n_].astype(np.float64)[None, :] if fco is not None else 1.0)
            bound = 0.5 * sg + 0.5 * so + (2.0 ** -10) * np.abs(So[n_]).max()
            worst = max(worst, float(np.max(np.abs(S[i, r % w.heads] - So[n_]) / bound)))
        return worst

    def code_mismatch(self):
        """INT8: (fraction of codes that differ, max |difference|) over sampled heads.

        Compensator pools: only codes whose quantization step (by the
        oracle's factors) is above 2^-18 of the state's magnitude are
        compared; below it the residual is the rounding left by the fitted
        pairs and its codes are not determined."""
        w, s = self.w, self.sample
        slots_b = self.slot_idx.cpu().numpy()[s.rows // w.heads]
        uniq = np.unique(slots_b)
        Z, sc = self.pool.read_int8(torch.as_tensor(uniq, dtype=torch.int32))
        Z = Z.cpu().numpy()
        pos = {int(x): i for i, x in enumerate(uniq)}
        Zo, so = self.orc.codes(s.state_idx)
        masks = None
        if self.compensators:
            step = so.astype(np.float64)[:, :, None] * np.ones((1, 1, D))
            if self.col_scales:
                step = step * self.orc.col_factors(s.state_idx).astype(np.float64)[:, None, :]
            mag = np.abs(self.orc.logical(s.state_idx)).reshape(len(s.rows), -1).max(axis=1)
            masks = step * 127.0 > (2.0 ** -18) * mag[:, None, None]
        diff = 0
        mx = 0
        count = 0
        for n_, r in enumerate(s.rows):
            d = np.abs(Z[pos[int(slots_b[n_])], r % w.heads].astype(np.int32) - Zo[n_].astype(np.int32))
            if masks is not None:
                d = d[masks[n_]]
            count += d.size
            diff += int((d > 0).sum())
            mx = max(mx, int(d.max()) if d.size else 0)
        return diff / max(count, 1), mx
