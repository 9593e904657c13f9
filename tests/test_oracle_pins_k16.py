"""Pins of the oracle's 16-bit key-side log factors ("DeltaLog: Deferred
Materialization of Recurrent States for Linear Attention Decoding", §3.4:
deferred key-side factors in 16-bit storage, value-side factors in FP32):
keys appended to the log are bfloat16 (FP32 rounded to its top 16 bits,
ties to even); reads of later tokens use the stored factor.
"""
import numpy as np
import pytest

from test_oracle_pins import DK, DV, GATES, make_inputs, relerr


def _bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def test_stored_keys_are_bfloat16_round_to_nearest(oracle_mod):
    rng = np.random.default_rng(90)
    n, M = 4, 8
    d = oracle_mod.DeferredOracle(n, DK, DV, 1, M, k16=True)
    q, k, v, lam, b = make_inputs(rng, M - 1, n, DK, 1, DV)
    for t in range(M - 1):
        d.step(range(n), q[t], k[t], v[t], lam[t], b[t])
    K = d.K[:, : M - 1].astype(np.float32)           # [n, M-1, DK]
    kin = np.transpose(k, (1, 0, 2))                 # [n, T, DK]
    assert np.all((_bits(K) & 0xFFFF) == 0)          # a bfloat16 value
    err = np.abs(K.astype(np.float64) - kin.astype(np.float64))
    assert np.all(err <= np.abs(kin) * 2.0 ** -8)    # half an ulp of an 8-bit significand
    assert np.any(err > 0)


def test_ties_round_to_even(oracle_mod):
    """1 + 2^-8 lies halfway between 1 and 1 + 2^-7 (odd): it goes to 1;
    1 + 3 2^-8 lies between 1 + 2^-7 (odd) and 1 + 2^-6 (even): it goes up."""
    d = oracle_mod.DeferredOracle(1, 4, 3, 1, 4, k16=True)
    k = np.array([[[1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.5]]], dtype=np.float32)
    z = np.zeros((1, 1, 4), np.float32)
    d.step([0], z[0], k[0], np.ones((1, 3), np.float32), np.zeros((1, 1), np.float32),
           np.ones(1, np.float32))
    assert list(d.K[0, 0]) == [1.0, 1 + 2 ** -6, -1.0, 0.5]


@pytest.mark.parametrize("gate,dl", GATES)
def test_bfloat16_exact_keys_change_nothing(oracle_mod, gate, dl):
    rng = np.random.default_rng(91)
    n, M, T = 3, 5, 13
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    k = (_bits(k) & 0xFFFF0000).view(np.float32)      # keys that bfloat16 holds exactly
    a = oracle_mod.DeferredOracle(n, DK, DV, dl, M)
    c = oracle_mod.DeferredOracle(n, DK, DV, dl, M, k16=True)
    for t in range(T):
        assert np.array_equal(a.step(range(n), q[t], k[t], v[t], lam[t], b[t]),
                              c.step(range(n), q[t], k[t], v[t], lam[t], b[t]))
    assert np.array_equal(a.logical(range(n)), c.logical(range(n)))


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_and_deferred_agree_on_stored_keys(oracle_mod, gate, dl):
    """Two separate implementations of "reads use the stored key": the
    window scheme (dense state corrected by (k^ - k) u^T after each token)
    with no quantization in the run, and the deferred scheme (base + log)
    with no merge in the run."""
    rng = np.random.default_rng(92)
    n, T = 3, 11
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=T + 1, k16=True)
    d = oracle_mod.DeferredOracle(n, DK, DV, dl, T + 2, k16=True)
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    for t in range(T):
        yw = w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        yd = d.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        ye = e.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        assert relerr(yw, yd) < 1e-12
        assert relerr(w.logical(range(n)), d.logical(range(n))) < 1e-12
    # and the stored keys move the trajectory by about their rounding
    diff = relerr(d.logical(range(n)), e.S)
    assert 1e-6 < diff < 2e-2
