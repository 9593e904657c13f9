"""Pins of the oracle's plain update rule: the update pair (k_t, v_t) with no
delta-rule correction, S_t = Diag(alpha_t) S_{t-1} + k_t v_t^T, y_t = S_t^T q_t
("DeltaLog: Deferred Materialization of Recurrent States for Linear
Attention Decoding", Table 1: the linear attention / RetNet / GLA / RWKV6
rows, with the post-update readout of eq. 3; "LeapQuant: Efficient Linear
Attention with Accurate Recurrent State Quantization", App. A with b_t = 0).
"""
import numpy as np
import pytest

from test_oracle_pins import DK, DV, GATES, make_inputs, relerr


def _alpha(lam, n, dk):
    return np.exp(np.broadcast_to(lam.astype(np.float64), (n, dk)))


@pytest.mark.parametrize("gate,dl", GATES)
def test_plain_matches_unrolled_closed_form(oracle_mod, gate, dl):
    """S_T = Gamma_{1:T} S_0 + sum_t Gamma_{t+1:T} k_t v_t^T with
    Gamma_{a:b} = prod of Diag(alpha) over tokens a..b."""
    rng = np.random.default_rng(80)
    n, T = 3, 9
    e = oracle_mod.EagerOracle(n, DK, DV, dl, plain=True)
    S0 = rng.standard_normal((n, DK, DV))
    e.load(range(n), S0)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    ys = [e.step(range(n), q[t], k[t], v[t], lam[t], b[t]) for t in range(T)]
    for t_end in range(T):
        G = np.ones((n, DK))
        S = np.zeros((n, DK, DV))
        for t in range(t_end, -1, -1):
            S += G[:, :, None] * np.einsum("ni,nj->nij", k[t].astype(np.float64), v[t].astype(np.float64))
            G = G * _alpha(lam[t], n, DK)
        S += G[:, :, None] * S0
        if t_end == T - 1:
            assert relerr(e.S, S) < 1e-12
        assert relerr(ys[t_end], np.einsum("nij,ni->nj", S, q[t_end].astype(np.float64))) < 1e-12


@pytest.mark.parametrize("gate,dl", GATES)
def test_plain_ignores_beta_and_is_linear_in_v(oracle_mod, gate, dl):
    rng = np.random.default_rng(81)
    n, T = 2, 7
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    v2 = rng.standard_normal(v.shape).astype(np.float32)

    def run(vv, bb):
        e = oracle_mod.EagerOracle(n, DK, DV, dl, plain=True)
        y = [e.step(range(n), q[t], k[t], vv[t], lam[t], bb[t]) for t in range(T)]
        return np.array(y), e.S.copy()

    y1, S1 = run(v, b)
    yb, Sb = run(v, np.zeros_like(b) + 0.123)
    assert np.array_equal(y1, yb) and np.array_equal(S1, Sb)
    y2, S2 = run(v2, b)
    y12, S12 = run((v.astype(np.float64) + v2).astype(np.float32), b)
    # exact in v up to the float32 rounding of v + v2
    assert relerr(S12, S1 + S2) < 1e-6 and relerr(y12, y1 + y2) < 1e-6
    # the delta rule is not linear in v (its correction reads the state)
    d = oracle_mod.EagerOracle(n, DK, DV, dl)
    for t in range(T):
        d.step(range(n), q[t], k[t], v[t], lam[t], b[t])
    assert relerr(d.S, S1) > 1e-3


def test_plain_without_decay_is_linear_attention(oracle_mod):
    """alpha = 1: S_T = sum_t k_t v_t^T and y_T = sum_t (k_t . q_T) v_t."""
    rng = np.random.default_rng(82)
    n, T = 2, 6
    q, k, v, lam, b = make_inputs(rng, T, n, DK, 1, DV)
    lam[:] = 0.0
    e = oracle_mod.EagerOracle(n, DK, DV, 1, plain=True)
    for t in range(T):
        y = e.step(range(n), q[t], k[t], v[t], lam[t], b[t])
    kk, vv, qq = (a.astype(np.float64) for a in (k, v, q[T - 1]))
    expect = np.einsum("tni,ni,tnj->nj", kk, qq, vv)
    assert relerr(y, expect) < 1e-12


@pytest.mark.parametrize("gate,dl", GATES)
@pytest.mark.parametrize("M", [1, 2, 5, 16])
def test_plain_deferred_equals_eager(oracle_mod, gate, dl, M):
    rng = np.random.default_rng(83)
    n, T = 3, 2 * M + 3
    e = oracle_mod.EagerOracle(n, DK, DV, dl, plain=True)
    d = oracle_mod.DeferredOracle(n, DK, DV, dl, M, plain=True)
    S0 = rng.standard_normal((n, DK, DV))
    e.load(range(n), S0)
    d.load(range(n), S0)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    for t in range(T):
        ye = e.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        yd = d.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        assert relerr(yd, ye) < 1e-12
        assert relerr(d.logical(range(n)), e.S) < 1e-12
