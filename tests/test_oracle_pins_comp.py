"""Pins of the oracle's Compensator Tokens ("LeapQuant: Efficient Linear
Attention with Accurate Recurrent State Quantization", §3.3 eq. 5-6, §3.4
eq. 7, App. B.3 eq. 10): r rank-one pairs fitted to the boundary state by
power iteration, kept in high precision, with only the residual quantized.

Pins: the exact rank-one case, the best rank-r approximation of a strongly
gapped spectrum (Eckart-Young: the truncated SVD), deflation leaving the
residual orthogonal to the last fitted direction, the accuracy gain the
method exists for, and the window forms (eq. 7 and eq. 10 with the pairs).
"""
import numpy as np
import pytest

from test_oracle_pins import DK, DV, GATES, make_inputs, relerr


def _gapped(rng, dk, dv, sig):
    U, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    V, _ = np.linalg.qr(rng.standard_normal((dv, dv)))
    s = np.zeros(min(dk, dv))
    s[:len(sig)] = sig
    return (U[:, :len(s)] * s) @ V[:, :len(s)].T


def test_rank_one_state_is_captured_exactly(oracle_mod):
    rng = np.random.default_rng(70)
    a, b = rng.standard_normal(12), rng.standard_normal(9) + 0.5
    S = np.outer(a, b)
    R, ck, cu = oracle_mod.fit_compensators(S, 1)
    assert relerr(np.outer(ck[0], cu[0]), S) < 1e-12
    assert np.max(np.abs(R)) <= 1e-12 * np.max(np.abs(S))
    assert abs(np.linalg.norm(cu[0]) - 1.0) < 1e-14


@pytest.mark.parametrize("r", [1, 2, 4])
def test_gapped_spectrum_matches_truncated_svd(oracle_mod, r):
    """With singular values 1e6, 1e4, 1e2, 1, ... three power steps per pair
    reach the top-r subspace: sum_h k~_h u~_h^T is the best rank-r
    approximation (the truncated SVD), and the residual is what is left."""
    rng = np.random.default_rng(71)
    S = _gapped(rng, 24, 20, [1e6, 1e4, 1e2, 1.0, 1e-2, 1e-3])
    R, ck, cu = oracle_mod.fit_compensators(S, r)
    U_, s_, Vt = np.linalg.svd(S)
    best = (U_[:, :r] * s_[:r]) @ Vt[:r]
    approx = np.einsum("hi,hj->ij", ck, cu)
    assert np.linalg.norm(approx - best) <= 1e-4 * np.linalg.norm(best)
    assert np.allclose(R, S - approx, atol=1e-9 * np.abs(S).max())
    assert np.allclose(np.linalg.norm(cu, axis=-1), 1.0, atol=1e-12)


def test_deflation_orthogonality(oracle_mod):
    """Each pair is k~ = R v, u~ = v on the residual left so far, so the final
    residual annihilates the last fitted direction: R u~_r = 0."""
    rng = np.random.default_rng(72)
    S = rng.standard_normal((16, 11)) * rng.uniform(0.1, 5.0, (16, 1))
    for r in (1, 3):
        R, ck, cu = oracle_mod.fit_compensators(S, r)
        assert np.max(np.abs(R @ cu[-1])) <= 1e-12 * np.abs(S).max() * 16
        assert np.allclose(R, S - np.einsum("hi,hj->ij", ck, cu), atol=1e-12 * np.abs(S).max())


def test_warm_start_on_the_singular_vector_is_a_fixed_point(oracle_mod):
    rng = np.random.default_rng(73)
    S = _gapped(rng, 10, 8, [5.0, 2.0, 1.0])
    _, _, Vt = np.linalg.svd(S)
    v1 = Vt[0]
    R, ck, cu = oracle_mod.fit_compensators(S, 1, warm_cu=v1[None, :])
    assert min(np.linalg.norm(cu[0] - v1), np.linalg.norm(cu[0] + v1)) < 1e-12


def test_compensators_cut_outlier_quantization_error(oracle_mod):
    """A state dominated by a rank-one outlier pattern: with the pair held in
    high precision the boundary state is far closer to the exact one."""
    rng = np.random.default_rng(74)
    n = 3
    S = rng.standard_normal((n, DK, DV)) * 0.05
    S += 40.0 * np.einsum("ni,nj->nij", rng.standard_normal((n, DK)), rng.standard_normal((n, DV)))
    err = {}
    for r in (0, 1):
        w = oracle_mod.WindowInt8Oracle(n, DK, DV, 1, W=4, compensators=r)
        w.load(range(n), S)
        err[r] = np.linalg.norm(w.logical(range(n)) - S)
    assert err[1] * 10 < err[0]


@pytest.mark.parametrize("cols", [False, True])
@pytest.mark.parametrize("gate,dl", GATES)
def test_window_of_one_with_compensators(oracle_mod, gate, dl, cols):
    """W = 1: every token ends a window: fit (cold start), quantize the
    residual, restart from dequant + K~ U~^T."""
    rng = np.random.default_rng(75)
    n, T, r = 2, 6, 2
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=1, col_scales=cols, compensators=r)
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    quant = oracle_mod.quantize_cols if cols else oracle_mod.quantize_rows
    deq = oracle_mod.dequantize_cols if cols else oracle_mod.dequantize_rows

    def boundary(S):
        R, ck, cu = oracle_mod.fit_compensators(S, r)
        q = quant(R)
        return deq(*q) + np.einsum("nhi,nhj->nij", ck, cu), q, cu

    S0 = rng.standard_normal((n, DK, DV))
    w.load(range(n), S0)
    S, q, cu = boundary(S0)
    assert np.array_equal(w.Z, q[0])
    assert relerr(w.logical(range(n)), S) < 1e-13
    e.load(range(n), S)
    q_, k_, v_, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    for t in range(T):
        yw = w.step(range(n), q_[t], k_[t], v_[t], lam[t], b[t])
        ye = e.step(range(n), q_[t], k_[t], v_[t], lam[t], b[t])
        assert relerr(yw, ye) < 1e-13
        S, q, cu = boundary(e.S)
        assert np.array_equal(w.Z, q[0])
        assert relerr(w.logical(range(n)), S) < 1e-12
        e.load(range(n), S)


@pytest.mark.parametrize("cols", [False, True])
@pytest.mark.parametrize("gate,dl", GATES)
def test_window_forms_with_compensators(oracle_mod, gate, dl, cols):
    """eq. 7 (the unrolled state) and eq. 10 (the readout, with the term
    U~ (K~^T Gamma x)) equal the recurrence at every position."""
    rng = np.random.default_rng(76)
    n, W, r = 2, 5, 3
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W, col_scales=cols, compensators=r)
    w.load(range(n), rng.standard_normal((n, DK, DV)) * 2.0)
    q, k, v, lam, b = make_inputs(rng, 2 * W + 2, n, DK, dl, DV)
    for t in range(2 * W + 2):
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        S = w.logical(range(n))
        assert relerr(w.unrolled(range(n)), S) < 1e-12
        x = rng.standard_normal((n, DK))
        assert relerr(w.readout(range(n), x), np.einsum("nij,ni->nj", S, x)) < 1e-12
    ck, cu = w.compensators(range(n))
    assert ck.shape == (n, r, DK) and np.allclose(np.linalg.norm(cu, axis=-1), 1.0)
