"""Pins of the oracle's smoothed per-value-column INT8 format ("LeapQuant:
Efficient Linear Attention with Accurate Recurrent State Quantization", §3.4
eq. 7 and App. B.3 eq. 10): key rows divided by the smoothing vector c (the
square root of each row's mean absolute value, floored), one symmetric INT8
scale per value column, dequantization C (Z / 127) B.

As in test_oracle_pins, no test compares the oracle with itself: each checks
an error bound, an exact invariance, a property the definition forces, a
degenerate case, or a second form the page gives for the same quantity.
States are non-square (d_k != d_v) so that a transposed factor fails.
"""
import numpy as np
import pytest

from test_oracle_pins import DK, DV, GATES, make_inputs, relerr

FLOOR = 2.0 ** -20


def _states(rng, n=4, dk=12, dv=20):
    """Rows and columns of very different magnitude, an outlier row and
    column (the structure smoothing is meant for), a zero row."""
    S = rng.standard_normal((n, dk, dv))
    S *= rng.uniform(0.01, 30.0, (n, dk, 1)) * rng.uniform(0.1, 10.0, (n, 1, dv))
    S[0, 2 % dk, :] *= 200.0
    S[1 % n, :, 5 % dv] *= 150.0
    S[2 % n, 4 % dk, :] = 0.0
    return S


def test_bound_and_column_absmax(oracle_mod):
    rng = np.random.default_rng(60)
    S = _states(rng)
    Z, c, b = oracle_mod.quantize_cols(S)
    assert Z.dtype == np.int8 and c.dtype == np.float32 and b.dtype == np.float32
    assert c.shape == S.shape[:-1] and b.shape == S.shape[:-2] + S.shape[-1:]
    assert Z.min() >= -127 and Z.max() <= 127
    Sf = S.astype(np.float32).astype(np.float64)
    deq = oracle_mod.dequantize_cols(Z, c, b)
    step = c.astype(np.float64)[..., :, None] * b.astype(np.float64)[..., None, :]
    # half a step, plus the FP32 roundings of 1/c, of S/c, of 127/B and B/127
    # and of the product
    bound = step * (0.5 + 128 * 2.0 ** -22) + np.abs(Sf) * 2.0 ** -21
    assert np.all(np.abs(deq - Sf) <= bound)
    # a wrong rounding direction would cost a whole step
    assert np.all(np.abs(deq - Sf) <= 0.51 * step + np.abs(Sf) * 2.0 ** -21 + 1e-30)
    # one scale per VALUE column: every nonzero column reaches +-127
    nzc = np.abs(S).max(axis=-2) > 0
    assert np.all(np.abs(Z).max(axis=-2)[nzc] == 127)
    # the zero row: floored smoothing factor, zero codes
    assert c[2, 4] == np.float32(FLOOR) and np.all(Z[2, 4] == 0)


def test_smoothing_balances_rows(oracle_mod):
    """With c_i^2 the row's mean |S_ij|, the smoothed row C^-1 S has mean
    absolute value c_i: rows of any magnitude come out at the square root of
    their magnitude (the balancing of §3.4).  A max- or rms-based c, or a c
    without the square root, fails this."""
    rng = np.random.default_rng(61)
    S = _states(rng)
    Z, c, b = oracle_mod.quantize_cols(S)
    deq = oracle_mod.dequantize_cols(Z, c, b)
    cd = c.astype(np.float64)
    smoothed_mean = np.abs(S / cd[..., None]).mean(axis=-1)
    live = np.abs(S).mean(axis=-1) > FLOOR ** 2
    assert np.allclose(smoothed_mean[live], cd[live], rtol=1e-6)
    # and the quantized state keeps that balance up to the quantization error
    assert np.allclose(np.abs(deq / cd[..., None]).mean(axis=-1)[live], cd[live], rtol=0.05)


@pytest.mark.parametrize("k", [-3, -1, 1, 2])
def test_exact_homogeneity(oracle_mod, k):
    """Scaling S by 4^k scales every row mean by 4^k exactly, c and b by 2^k
    exactly, and leaves every code unchanged (all FP32 operations on the
    scaled values are exact images of the unscaled ones)."""
    rng = np.random.default_rng(62)
    S = _states(rng)
    S[2, 4, :] = rng.standard_normal(S.shape[-1])  # no floored row here
    Z, c, b = oracle_mod.quantize_cols(S)
    Zk, ck, bk = oracle_mod.quantize_cols(S * 4.0 ** k)
    assert np.array_equal(Zk, Z)
    assert np.array_equal(ck, c * np.float32(2.0 ** k))
    assert np.array_equal(bk, b * np.float32(2.0 ** k))


def test_degenerate_columns_and_state(oracle_mod):
    Z, c, b = oracle_mod.quantize_cols(np.zeros((3, 7)))
    assert np.all(Z == 0) and np.all(b == 0) and np.all(c == np.float32(FLOOR))
    # every |S_ij| = 1: every row mean is 1, so c = 1 exactly and every code 127
    Z, c, b = oracle_mod.quantize_cols(np.ones((3, 7)))
    assert np.all(c == 1.0) and np.all(b == np.float32(1.0) / np.float32(127.0))
    assert np.all(Z == 127)
    # a zero column: scale 0 and zero codes there, the others untouched
    S = np.ones((3, 7))
    S[:, 2] = 0.0
    Z, c, b = oracle_mod.quantize_cols(S)
    assert b[2] == 0 and np.all(Z[:, 2] == 0)
    assert np.all(Z[:, [0, 1, 3, 4, 5, 6]] == 127)


# --------------------------------------------------------------------------
# the per-window scheme in the smoothed format
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gate,dl", GATES)
def test_window_of_one_is_per_step_smoothed_quantization(oracle_mod, gate, dl):
    rng = np.random.default_rng(63)
    n, T = 3, 10
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=1, col_scales=True)
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    S0 = rng.standard_normal((n, DK, DV))
    w.load(range(n), S0)
    Z0, c0, b0 = oracle_mod.quantize_cols(S0)
    assert np.array_equal(w.Z, Z0) and np.array_equal(w.s, c0)
    assert np.array_equal(w.col_factors(range(n)), b0)
    e.load(range(n), oracle_mod.dequantize_cols(Z0, c0, b0))
    q, k, v, lam, bb = make_inputs(rng, T, n, DK, dl, DV)
    for t in range(T):
        yw = w.step(range(n), q[t], k[t], v[t], lam[t], bb[t])
        ye = e.step(range(n), q[t], k[t], v[t], lam[t], bb[t])
        assert np.array_equal(yw, ye)
        Z, c, b = oracle_mod.quantize_cols(e.S)
        assert np.array_equal(w.Z, Z) and np.array_equal(w.s, c)
        assert np.array_equal(w.col_factors(range(n)), b)
        e.load(range(n), oracle_mod.dequantize_cols(Z, c, b))


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_unrolled_and_readout_eq10(oracle_mod, gate, dl):
    """In the smoothed format the in-window state is eq. 7's S_l and its
    readout B Z^T C Gamma x / 127 + records (eq. 10) equals S_l^T x."""
    rng = np.random.default_rng(64)
    n, W = 3, 6
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W, col_scales=True)
    w.load(range(n), _states(rng, n, DK, DV))
    q, k, v, lam, b = make_inputs(rng, 2 * W + 2, n, DK, dl, DV)
    for t in range(2 * W + 2):
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        S = w.logical(range(n))
        assert relerr(w.unrolled(range(n)), S) < 1e-12
        x = rng.standard_normal((n, DK))
        assert relerr(w.readout(range(n), x), np.einsum("nij,ni->nj", S, x)) < 1e-12


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_longer_than_run_is_eager_smoothed(oracle_mod, gate, dl):
    rng = np.random.default_rng(65)
    n, T = 2, 9
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=T + 1, col_scales=True)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    for t in range(T):
        ye = e.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        yw = w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        assert relerr(yw, ye) < 1e-13


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_commit_smoothed(oracle_mod, gate, dl):
    rng = np.random.default_rng(66)
    n, W = 3, 5
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W, col_scales=True)
    w.load(range(n), rng.standard_normal((n, DK, DV)))
    q, k, v, lam, b = make_inputs(rng, 3, n, DK, dl, DV)
    for t in range(3):
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
    S_mid = w.logical(range(n))
    w.commit([0])
    Z, c, bc = oracle_mod.quantize_cols(S_mid[0])
    assert np.array_equal(w.Z[0], Z) and np.array_equal(w.s[0], c)
    assert np.array_equal(w.col_factors([0])[0], bc)
    assert list(w.cnt) == [0, 3, 3]


def test_column_rounding_is_half_to_even(oracle_mod):
    """Every row has mean |S| = 1, so c = 1 exactly; column 0's absmax is
    127/64, so its factor 127/B is 64 exactly and +-5/128 lands on +-2.5."""
    S = np.array([[127 / 64, 1 / 64], [5 / 128, 251 / 128], [-5 / 128, 251 / 128]])
    Z, c, b = oracle_mod.quantize_cols(S)
    assert np.all(c == 1.0)
    assert list(Z[:, 0]) == [127, 2, -2]
    assert b[0] == np.float32(127 / 64) / np.float32(127.0)
