"""Compensator Tokens on the GPU against what the page fixes about them.

"LeapQuant: Efficient Linear Attention with Accurate Recurrent State
Quantization", §3.3 eq. 5-6: at a window boundary r rank-one pairs are
fitted to the state, so that only the residual S - K~ U~^T is quantized.
The best rank-r pairs are the truncated SVD (Eckart-Young): no rank-r
product removes more of ||S||_F^2 than the r largest squared singular
values.  The fit itself (power iteration, three steps per pair) is a
reading of the page, so beyond that bound these tests hold the GPU's own
pairs to what the fit and the quantizer must give for the state they see:

  1. energy: E(X) = ||S||^2 - ||S - X||^2 for X the GPU's K~ U~^T satisfies
     E(X) <= sum_{h<r} sigma_h^2 (Eckart-Young, with room for the double
     rounding of the check), and E(X) >= (1 - ENERGY_TOL) E(X_o), X_o the
     oracle's fit of the same S.  ENERGY_TOL = 1e-3: the GPU fits an FP32
     copy of S (about 1e-6 relative to it after a window of FP32 updates)
     with FP32 arithmetic, and pair h carries that rounding amplified by
     sigma_1 / sigma_h through the deflations; E is first-order in the
     pairs, so its relative change is at most the pairs' (products within
     1e-3 of the oracle's on these states, as the parity tests check);
  2. residual: the GPU's dequantized codes equal S - X (its own pairs) within
     half its own code step (the quantizer's bound, with the FP32 rounding
     of the step and factor) plus 2^-16 max|S| for the FP32 state it fitted
     and quantized.

S is the oracle's: each workload's input law and shapes, one window from the
zero state (both sides hold it exactly, pairs k~ = 0), so the unquantized
boundary state is the plain recurrence over the window, computed by the
eager oracle for a sample of heads; no GPU value enters the oracle.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

R = 4
ENERGY_TOL = 1e-3
STATE_SLACK = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _window_end(name, W, cols, n_sample, seed=5):
    import _harness as H
    import oracle
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import workloads as wl
    base = wl.WORKLOAD_BY_NAME[name]
    w = wl.Workload(**{**base.__dict__, "pools": 1, "prewarm_tokens": 0})
    dev = torch.device("cuda")
    pool = StatePool(w.num_slots, w.heads, "int8", w.gate, W, device=dev, col_scales=cols,
                     compensators=R)
    slot_idx = wl.slot_index(w, dev)
    masks = wl.static_masks(w, dev)
    s = H.sample_rows(w, slot_idx, n_sample, seed)
    eag = oracle.EagerOracle(len(s.rows), H.D, H.D, w.dl)
    idx = np.arange(len(s.rows))
    for t in range(W):  # the W-th token closes the first window
        ins = wl.step_inputs(w, t, device=dev, masks=masks)
        pool.decode_step(slot_idx, *ins)
        eag.step(idx, *H.host_inputs(ins, w, s.rows))
    S = eag.logical(idx)
    slots = slot_idx.cpu().numpy()[s.rows // w.heads]
    heads = s.rows % w.heads
    uniq = np.unique(slots)
    ut = torch.as_tensor(uniq, dtype=torch.int32, device=dev)
    kk, uu = (x.double().cpu().numpy() for x in pool.read_compensators(ut))
    Z, fr = pool.read_int8(ut)
    Z, fr = Z.cpu().numpy().astype(np.float64), fr.double().cpu().numpy()
    fc = pool.read_int8_col_scales(ut).double().cpu().numpy() if cols else None
    ln, _ = pool.read_log_meta(ut)
    assert torch.all(ln == R), "a window end leaves the r new pairs at the head of the log"
    assert pool.status() == 0
    pos = {int(x): i for i, x in enumerate(uniq)}
    out = []
    for n_ in range(len(s.rows)):
        i, h = pos[int(slots[n_])], int(heads[n_])
        col = fc[i, h][None, :] if cols else 1.0
        out.append((S[n_], kk[i, h], uu[i, h], Z[i, h], fr[i, h][:, None] * col))
    return out


def _energy(S, X):
    return float((S * S).sum() - ((S - X) ** 2).sum())


@pytest.mark.parametrize("name,W,cols,n_sample", [
    ("kda_b128_h32_t512_longlived", 32, True, 6),
    ("kda_b128_h32_t512_longlived", 32, False, 4),
    ("gdn_serving_b256_h48_4pools", 16, True, 6),
    ("gdn_serving_b256_h48_4pools", 16, False, 4),
])
def test_pairs_capture_the_truncated_svd_energy_and_leave_the_quantized_residual(name, W, cols, n_sample):
    import oracle
    ratios = []
    for S, kk, uu, Z, step in _window_end(name, W, cols, n_sample):
        X = np.einsum("hi,hj->ij", kk, uu)
        sig = np.linalg.svd(S, compute_uv=False)
        e_svd = float((sig[:R] ** 2).sum())
        e_gpu = _energy(S, X)
        _, ko, uo = oracle.fit_compensators(S, R)
        e_orc = _energy(S, np.einsum("hi,hj->ij", ko, uo))
        norm2 = float((S * S).sum())
        # Eckart-Young: no rank-r product captures more than the truncated SVD
        assert e_gpu <= e_svd * (1 + 1e-9) + 1e-12 * norm2, (e_gpu, e_svd)
        assert e_orc <= e_svd * (1 + 1e-9) + 1e-12 * norm2, (e_orc, e_svd)
        # the GPU's fit captures what the fit of the same state does
        assert e_gpu >= (1 - ENERGY_TOL) * e_orc, (e_gpu, e_orc)
        ratios.append(e_gpu / e_svd)
        # the codes are the residual the GPU's own pairs leave, quantized
        bound = step * (0.5 + 128 * 2.0 ** -22) + STATE_SLACK * np.abs(S).max()
        err = np.abs(step * Z - (S - X)) / bound
        assert float(err.max()) <= 1.0, float(err.max())
    print(f"{name} W={W} cols={cols}: captured / truncated-SVD energy "
          f"{min(ratios):.4f}..{max(ratios):.4f}")
