"""Pins of the oracle's FP16 records ("LeapQuant: Efficient Linear Attention
with Accurate Recurrent State Quantization", §4.3: the window's buffered
records (k, u) and the compensator pairs are kept in FP16): values rounded
to the nearest IEEE binary16 number, ties to even; the current token's own
output uses k and u themselves, later reads use the stored records.

numpy's float16 conversion (round to nearest even, with subnormals) is the
independent reference for the rounding.
"""
import numpy as np
import pytest

from test_oracle_pins import DK, DV, GATES, make_inputs, relerr


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def test_stored_keys_are_binary16_incl_ties_subnormals_and_range(oracle_mod):
    """beta = 0 keeps u = 0, so crafted keys only exercise the rounding:
    ties (1 + 2^-11 -> 1, 1 + 3 2^-11 -> 1 + 2^-9), subnormals (spacing 2^-24,
    2^-25 is a tie -> 0, 3 2^-26 -> 2^-24), the largest finite value and a
    value just below the overflow threshold (65519 -> 65504)."""
    vals = [1 + 2 ** -11, 1 + 3 * 2 ** -11, -(1 + 2 ** -11), 2.0 ** -25, 3 * 2.0 ** -26,
            1e-6, -7.3e-7, 65504.0, 65519.0, 0.1, -0.3, 2.0 ** -14 * 1.5]
    dk = len(vals)
    w = oracle_mod.WindowInt8Oracle(1, dk, 3, 1, W=8, r16=True)
    k = np.array([[vals]], dtype=np.float32)
    z = np.zeros((1, 1, dk), np.float32)
    w.step([0], z[0], k[0], np.ones((1, 3), np.float32), np.zeros((1, 1), np.float32),
           np.zeros(1, np.float32))
    got = w.rk[0, 0]
    assert np.array_equal(got, _f16(k[0, 0]))
    assert got[0] == 1.0 and got[1] == 1 + 2 ** -9 and got[3] == 0.0 and got[4] == 2.0 ** -24
    assert got[8] == 65504.0


@pytest.mark.parametrize("gate,dl", GATES)
def test_records_are_the_binary16_of_the_fp32_records(oracle_mod, gate, dl):
    """From one loaded state the FP32-record and FP16-record schemes compute
    the same first token (rounding happens at the append), and store the
    same record, rounded."""
    rng = np.random.default_rng(120)
    n = 4
    S0 = rng.standard_normal((n, DK, DV))
    a = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=6)
    b = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=6, r16=True)
    a.load(range(n), S0)
    b.load(range(n), S0)
    q, k, v, lam, bb = make_inputs(rng, 1, n, DK, dl, DV)
    ya = a.step(range(n), q[0], k[0], v[0], lam[0], bb[0])
    yb = b.step(range(n), q[0], k[0], v[0], lam[0], bb[0])
    assert np.array_equal(ya, yb)
    assert np.array_equal(b.rk[:, 0], _f16(a.rk[:, 0]))
    assert np.array_equal(b.ru[:, 0], _f16(a.ru[:, 0]))
    assert np.any(b.ru[:, 0] != a.ru[:, 0])
    # the state now holds the stored record: it differs from the FP32-record
    # state by exactly k^ u^T - k u^T
    dlt = (np.einsum("ni,nj->nij", b.rk[:, 0], b.ru[:, 0])
           - np.einsum("ni,nj->nij", a.rk[:, 0], a.ru[:, 0]))
    assert relerr(b.logical(range(n)) - a.logical(range(n)), dlt) < 1e-9


@pytest.mark.parametrize("gate,dl", GATES)
@pytest.mark.parametrize("cols", [False, True])
def test_unrolled_window_equals_incremental_state(oracle_mod, gate, dl, cols):
    """eq. 4 rebuilt from the boundary state and the stored FP16 records
    equals the state the recurrence carries (which applies the
    record-rounding correction token by token), and so does the eq. 9 / 10
    readout."""
    rng = np.random.default_rng(121)
    n, W = 3, 7
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W, col_scales=cols, r16=True)
    w.load(range(n), rng.standard_normal((n, DK, DV)))
    q, k, v, lam, b = make_inputs(rng, 2 * W + 3, n, DK, dl, DV)
    for t in range(2 * W + 3):
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        S = w.logical(range(n))
        assert relerr(w.unrolled(range(n)), S) < 1e-12
        x = rng.standard_normal((n, DK))
        assert relerr(w.readout(range(n), x), np.einsum("nij,ni->nj", S, x)) < 1e-12


@pytest.mark.parametrize("gate,dl", GATES)
def test_beta_zero_reduces_to_fp32_records(oracle_mod, gate, dl):
    """With beta = 0 every record is (k, 0): the rounded key multiplies a
    zero vector, so the FP16 scheme follows the FP32 one bit for bit."""
    rng = np.random.default_rng(122)
    n, W, T = 3, 5, 17
    a = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W)
    b = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W, r16=True)
    S0 = rng.standard_normal((n, DK, DV))
    a.load(range(n), S0)
    b.load(range(n), S0)
    q, k, v, lam, bb = make_inputs(rng, T, n, DK, dl, DV)
    zero = np.zeros_like(bb)
    for t in range(T):
        assert np.array_equal(a.step(range(n), q[t], k[t], v[t], lam[t], zero[t]),
                              b.step(range(n), q[t], k[t], v[t], lam[t], zero[t]))
    assert np.array_equal(a.logical(range(n)), b.logical(range(n)))
    assert np.array_equal(a.Z, b.Z)


@pytest.mark.parametrize("cols", [False, True])
def test_fp16_compensator_pairs(oracle_mod, cols):
    """The pairs are stored in FP16; the codes are the quantization of what
    the stored (rounded) pairs leave of the state, and the restart state is
    the dequantized residual plus the stored pairs."""
    rng = np.random.default_rng(123)
    n, r = 3, 4
    S = rng.standard_normal((n, DK, DV))
    S += 8.0 * np.einsum("ni,nj->nij", rng.standard_normal((n, DK)), rng.standard_normal((n, DV)))
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, 1, W=4, col_scales=cols, compensators=r,
                                    r16=True)
    w.load(range(n), S)
    ck, cu = w.compensators(range(n))
    assert np.array_equal(ck, _f16(ck)) and np.array_equal(cu, _f16(cu))
    R = S - np.einsum("nhi,nhj->nij", ck, cu)
    if cols:
        Z, c, bcol = oracle_mod.quantize_cols(R)
        assert np.array_equal(w.Z, Z) and np.array_equal(w.s, c)
        assert np.array_equal(w.col_factors(range(n)), bcol)
        deq = oracle_mod.dequantize_cols(Z, c, bcol)
    else:
        Z, s = oracle_mod.quantize_rows(R)
        assert np.array_equal(w.Z, Z) and np.array_equal(w.s, s)
        deq = oracle_mod.dequantize_rows(Z, s)
    assert relerr(w.logical(range(n)), deq + np.einsum("nhi,nhj->nij", ck, cu)) < 1e-12
    # the rounded pairs still take the dominant rank-one part out
    assert np.linalg.norm(R) < 0.5 * np.linalg.norm(S)


def test_fp16_and_bfloat16_records_are_exclusive(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.WindowInt8Oracle(1, DK, DV, 1, W=4, k16=True, r16=True)
