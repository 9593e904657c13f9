"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

None of these tests compares the oracle with itself: each one checks it
against a closed form, a special case, a second formula the pages state for the
same quantity, an invariant, or an error bound.  States are non-square
(d_k != d_v) wherever possible so that a transposed operand fails.

Pages: "LeapQuant: Efficient Linear Attention with Accurate Recurrent State
Quantization" (App. A product and expanded forms, §3.2 eq. 2-4, App. B.1
eq. 8, App. B.2 eq. 9, App. B.3) and "DeltaLog: Deferred Materialization of
Recurrent States for Linear Attention Decoding" (§3.1 Algorithm 1, §3.2 eq. 7
and its closure argument).
"""
import numpy as np
import pytest

DK, DV = 6, 5


def softplus(x):
    return np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0)


def make_inputs(rng, T, n, dk, dl, dv, lam_scale=0.3, beta=None, unit_k=True):
    q = rng.standard_normal((T, n, dk))
    k = rng.standard_normal((T, n, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, n, dv))
    lam = -softplus(rng.standard_normal((T, n, dl))) * lam_scale
    b = rng.uniform(0.0, 1.0, (T, n)) if beta is None else np.full((T, n), beta)
    f = lambda a: a.astype(np.float32)
    return f(q), f(k), f(v), f(lam), f(b)


def relerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / (den if den > 0 else 1.0))


GATES = [("gdn", 1), ("kda", DK)]


# --------------------------------------------------------------------------
# eager recurrence
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gate,dl", GATES)
def test_beta_zero_no_decay_leaves_state(oracle_mod, gate, dl):
    """beta = 0 and D = I: S is unchanged and y = S^T q (LeapQuant eq. 1)."""
    rng = np.random.default_rng(1)
    n = 3
    o = oracle_mod.EagerOracle(n, DK, DV, dl)
    S0 = rng.standard_normal((n, DK, DV))
    o.load(range(n), S0)
    q, k, v, lam, b = make_inputs(rng, 4, n, DK, dl, DV, beta=0.0)
    lam[:] = 0.0
    for t in range(4):
        y = o.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        assert np.array_equal(o.S, S0)
        assert relerr(y, np.einsum("nij,ni->nj", S0, q[t].astype(np.float64))) < 1e-14


@pytest.mark.parametrize("gate,dl", GATES)
def test_unit_key_beta_one_overwrites_along_key(oracle_mod, gate, dl):
    """||k|| = 1, beta = 1, D = I: k^T S_t = v_t (the delta rule writes v along k)."""
    rng = np.random.default_rng(2)
    n = 4
    o = oracle_mod.EagerOracle(n, DK, DV, dl)
    o.load(range(n), rng.standard_normal((n, DK, DV)))
    q, k, v, lam, b = make_inputs(rng, 6, n, DK, dl, DV, beta=1.0)
    lam[:] = 0.0
    # keys with four entries +-1/2 have norm exactly 1 in binary floating point
    k[:] = 0.0
    for t in range(6):
        for r in range(n):
            pos = rng.choice(DK, 4, replace=False)
            k[t, r, pos] = rng.choice([-0.5, 0.5], 4)
    for t in range(6):
        o.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        kS = np.einsum("ni,nij->nj", k[t].astype(np.float64), o.S)
        assert relerr(kS, v[t]) < 1e-13
    # basis key: row m of S becomes v
    e = np.zeros((n, DK), np.float32)
    e[:, 2] = 1.0
    o.step(range(n), q[0], e, v[0], lam[0], b[0])
    assert relerr(o.S[:, 2, :], v[0]) < 1e-14


@pytest.mark.parametrize("gate,dl", GATES)
def test_beta_zero_is_pure_decay(oracle_mod, gate, dl):
    """beta = 0: S_T = Gamma_{1:T} S_0 with Gamma the product of the decays."""
    rng = np.random.default_rng(3)
    n, T = 3, 9
    o = oracle_mod.EagerOracle(n, DK, DV, dl)
    S0 = rng.standard_normal((n, DK, DV))
    o.load(range(n), S0)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV, beta=0.0, lam_scale=0.7)
    cum = np.zeros((n, DK))
    for t in range(T):
        y = o.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        cum += np.broadcast_to(lam[t].astype(np.float64), (n, DK)) if dl == 1 else lam[t]
        expect = np.exp(cum)[:, :, None] * S0
        assert relerr(o.S, expect) < 1e-13
        assert relerr(y, np.einsum("nij,ni->nj", expect, q[t].astype(np.float64))) < 1e-13


@pytest.mark.parametrize("gate,dl", GATES)
def test_matches_product_form(oracle_mod, gate, dl):
    """The oracle's expanded form equals the product form of LeapQuant App. A:
    GDN  alpha (I - beta k k^T) S + beta k v^T,
    KDA  (I - beta k k^T) Diag(alpha) S + beta k v^T,  y = S^T q."""
    rng = np.random.default_rng(4)
    n, T = 2, 25
    o = oracle_mod.EagerOracle(n, DK, DV, dl)
    S0 = rng.standard_normal((n, DK, DV))
    o.load(range(n), S0)
    S = S0.copy()
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV, unit_k=False)
    I = np.eye(DK)
    for t in range(T):
        y = o.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        for r in range(n):
            kk = k[t, r].astype(np.float64)
            bb = float(b[t, r])
            P = I - bb * np.outer(kk, kk)
            if dl == 1:
                S[r] = np.exp(float(lam[t, r, 0])) * (P @ S[r]) + bb * np.outer(kk, v[t, r])
            else:
                D = np.diag(np.exp(lam[t, r].astype(np.float64)))
                S[r] = P @ D @ S[r] + bb * np.outer(kk, v[t, r])
        assert relerr(o.S, S) < 1e-12
        assert relerr(y, np.einsum("nij,ni->nj", S, q[t].astype(np.float64))) < 1e-12


def test_scalar_gate_equals_equal_per_key_gates(oracle_mod):
    """KDA with all per-key gates equal is Gated DeltaNet (App. A rows coincide)."""
    rng = np.random.default_rng(5)
    n, T = 3, 12
    g = oracle_mod.EagerOracle(n, DK, DV, 1)
    kd = oracle_mod.EagerOracle(n, DK, DV, DK)
    S0 = rng.standard_normal((n, DK, DV))
    g.load(range(n), S0)
    kd.load(range(n), S0)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, 1, DV)
    for t in range(T):
        y1 = g.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        y2 = kd.step(range(n), q[t], k[t], v[t], np.repeat(lam[t], DK, axis=1), b[t])
        assert np.array_equal(y1, y2)
    assert np.array_equal(g.S, kd.S)


@pytest.mark.parametrize("gate,dl", GATES)
def test_transition_is_a_contraction(oracle_mod, gate, dl):
    """With ||k|| = 1, beta in [0,1] and 0 < D <= I the state transition has
    spectral norm <= 1 (the property the STEPQuant notes and LeapQuant App. B.1
    rely on), so two trajectories fed the same tokens never move apart."""
    rng = np.random.default_rng(6)
    n, T = 4, 40
    a = oracle_mod.EagerOracle(n, DK, DV, dl)
    c = oracle_mod.EagerOracle(n, DK, DV, dl)
    a.load(range(n), rng.standard_normal((n, DK, DV)))
    c.load(range(n), rng.standard_normal((n, DK, DV)))
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV, lam_scale=0.05)
    b[:] = np.maximum(b, 0.5)
    prev = np.linalg.norm(a.S - c.S, axis=(1, 2))
    start = prev.copy()
    for t in range(T):
        a.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        c.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        cur = np.linalg.norm(a.S - c.S, axis=(1, 2))
        assert np.all(cur <= prev * (1 + 1e-12))
        prev = cur
    # and it does contract: beta >= 0.5 along ever-changing keys
    assert np.all(prev < 0.5 * start)


# --------------------------------------------------------------------------
# deferred materialization
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gate,dl", GATES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 16])
def test_deferred_equals_eager(oracle_mod, gate, dl, M):
    """DeltaLog's closure argument: base + log represents the eager state at
    every step in exact arithmetic, for every merge interval."""
    rng = np.random.default_rng(10 + M)
    n, T = 3, 37
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    d = oracle_mod.DeferredOracle(n, DK, DV, dl, M)
    S0 = rng.standard_normal((n, DK, DV))
    e.load(range(n), S0)
    d.load(range(n), S0)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    perm = np.array([2, 0, 1])
    for t in range(T):
        idx = perm if t % 2 else np.arange(n)
        ye = e.step(idx, q[t], k[t], v[t], lam[t], b[t])
        yd = d.step(idx, q[t], k[t], v[t], lam[t], b[t])
        if M == 1:
            assert np.array_equal(ye, yd)
        else:
            assert relerr(yd, ye) < 1e-12
        assert relerr(d.logical(range(n)), e.S) < 1e-12
        assert np.all(d.L == (t + 1) % M)
    if M == 1:
        assert np.array_equal(d.base, e.S)


@pytest.mark.parametrize("gate,dl", GATES)
def test_deferred_explicit_commit(oracle_mod, gate, dl):
    rng = np.random.default_rng(20)
    n, M = 3, 6
    d = oracle_mod.DeferredOracle(n, DK, DV, dl, M)
    d.load(range(n), rng.standard_normal((n, DK, DV)))
    q, k, v, lam, b = make_inputs(rng, 4, n, DK, dl, DV)
    for t in range(4):
        d.step(range(n), q[t], k[t], v[t], lam[t], b[t])
    before = d.logical(range(n))
    d.commit([0, 2])
    assert list(d.L) == [0, 4, 0]
    assert np.all(d.lbar[[0, 2]] == 0)
    assert relerr(d.logical(range(n)), before) < 1e-13
    base_before = d.base.copy()
    d.commit([0])  # empty log: nothing to fold
    assert np.array_equal(d.base, base_before)


# --------------------------------------------------------------------------
# INT8 quantizer
# --------------------------------------------------------------------------

def test_quantizer_bounds_and_idempotence(oracle_mod):
    rng = np.random.default_rng(30)
    S = rng.standard_normal((5, 16, 40)) * rng.uniform(0.01, 100.0, (5, 16, 1))
    S[1, 3, :] = 0.0
    S[2, 7, 11] = 1e4  # an outlier row
    Z, s = oracle_mod.quantize_rows(S)
    assert Z.dtype == np.int8 and s.dtype == np.float32
    assert Z.min() >= -127 and Z.max() <= 127
    Sf = S.astype(np.float32).astype(np.float64)
    deq = oracle_mod.dequantize_rows(Z, s)
    # half a step, plus the FP32 rounding of the factor 127 / absmax and of the
    # product (at most 128 * 2^-23 of a step) and of S itself
    sd = s.astype(np.float64)[..., None]
    bound = sd * (0.5 + 128 * 2.0 ** -22) + np.abs(Sf) * 2.0 ** -22
    assert np.all(np.abs(deq - Sf) <= bound)
    # never more than half a step plus rounding: a wrong rounding direction
    # would cost a whole step
    assert np.all(np.abs(deq - Sf) <= 0.51 * sd + 1e-30)
    nz = np.abs(S).max(axis=-1) > 0
    assert np.all(np.abs(Z).max(axis=-1)[nz] == 127)
    assert s[1, 3] == 0 and np.all(Z[1, 3] == 0)
    Z2, s2 = oracle_mod.quantize_rows(deq)
    assert np.array_equal(Z2, Z)
    assert np.all(np.abs(s2.astype(np.float64) - s) <= np.spacing(s))


def test_quantizer_rounds_half_to_even(oracle_mod):
    row = np.array([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, 126.5, 0.0])
    Z, s = oracle_mod.quantize_rows(row[None, :])
    assert s[0] == 1.0
    assert list(Z[0]) == [127, 2, 4, -2, -4, 0, 2, 0, 126, 0]
    # absmax 254: factor 127/254 = 0.5 exactly, so 5.0 -> 2.5 -> 2 and 7.0 -> 3.5 -> 4
    Z, s = oracle_mod.quantize_rows(np.array([[254.0, 5.0, 7.0, -5.0, 1.0]]))
    assert s[0] == np.float32(254.0) / np.float32(127.0)
    assert list(Z[0]) == [127, 2, 4, -2, 0]


def test_quantizer_degenerate_rows(oracle_mod):
    tiny = np.float32(1e-38) / np.float32(1e4)  # subnormal: 127 / absmax overflows FP32
    Z, s = oracle_mod.quantize_rows(np.array([[0.0, 0.0, 0.0], [tiny, -tiny, 0.0]]))
    assert np.all(s == 0) and np.all(Z == 0)


# --------------------------------------------------------------------------
# per-window INT8 scheme
# --------------------------------------------------------------------------

@pytest.mark.parametrize("gate,dl", GATES)
def test_window_longer_than_run_is_eager(oracle_mod, gate, dl):
    """A zero start state is exactly representable; with W > T nothing is
    quantized again, so the per-window trajectory is the eager one."""
    rng = np.random.default_rng(40)
    n, T = 3, 15
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=T + 1)
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    for t in range(T):
        ye = e.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        yw = w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        assert relerr(yw, ye) < 1e-13
    assert relerr(w.logical(range(n)), e.S) < 1e-13
    assert np.all(w.Z == 0)


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_of_one_is_per_step_quantization(oracle_mod, gate, dl):
    """W = 1 reduces to LeapQuant eq. 2: update from the quantized state, then
    quantize the result after every token."""
    rng = np.random.default_rng(41)
    n, T = 3, 12
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=1)
    e = oracle_mod.EagerOracle(n, DK, DV, dl)
    S0 = rng.standard_normal((n, DK, DV))
    w.load(range(n), S0)
    Z0, s0 = oracle_mod.quantize_rows(S0)
    e.load(range(n), oracle_mod.dequantize_rows(Z0, s0))
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV)
    for t in range(T):
        yw = w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        ye = e.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        assert np.array_equal(yw, ye)
        Z, s = oracle_mod.quantize_rows(e.S)
        assert np.array_equal(w.Z, Z) and np.array_equal(w.s, s)
        e.load(range(n), oracle_mod.dequantize_rows(Z, s))


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_unrolled_and_readout_forms(oracle_mod, gate, dl):
    """The in-window state equals eq. 4 (boundary state + records) and its
    readout equals eq. 9 (no d_k x d_v intermediate), at every position."""
    rng = np.random.default_rng(42)
    n, W = 3, 7
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W)
    w.load(range(n), rng.standard_normal((n, DK, DV)) * 3.0)
    q, k, v, lam, b = make_inputs(rng, 2 * W + 3, n, DK, dl, DV)
    for t in range(2 * W + 3):
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        S = w.logical(range(n))
        assert relerr(w.unrolled(range(n)), S) < 1e-12
        x = rng.standard_normal((n, DK))
        assert relerr(w.readout(range(n), x), np.einsum("nij,ni->nj", S, x)) < 1e-12
        assert np.all(w.cnt == (t + 1) % W)


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_error_recursion_and_bound(oracle_mod, gate, dl):
    """LeapQuant App. B.1 eq. 8: E_t = D_t E_{t-1} - k (E_{t-1}^T b)^T + eps_t
    with b = beta (alpha . k), eps_t nonzero only at window boundaries; and,
    the transition being a contraction, ||E_T||_F <= sum_s ||eps_s||_F."""
    rng = np.random.default_rng(43)
    n, W, T = 3, 4, 22
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W)
    fp = oracle_mod.EagerOracle(n, DK, DV, dl)
    pre = oracle_mod.EagerOracle(n, DK, DV, dl)
    S0 = rng.standard_normal((n, DK, DV))
    w.load(range(n), S0)
    fp.load(range(n), w.logical(range(n)))  # E_0 = 0
    q, k, v, lam, b = make_inputs(rng, T, n, DK, dl, DV, lam_scale=0.05)
    E = np.zeros((n, DK, DV))
    eps_sum = np.zeros(n)
    for t in range(T):
        pre.load(range(n), w.logical(range(n)))
        pre.step(range(n), q[t], k[t], v[t], lam[t], b[t])  # unquantized S_t
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        fp.step(range(n), q[t], k[t], v[t], lam[t], b[t])
        eps = w.logical(range(n)) - pre.S
        if (t + 1) % W:
            assert np.all(eps == 0)
        alpha = np.exp(np.broadcast_to(lam[t].astype(np.float64), (n, DK)))
        kk = k[t].astype(np.float64)
        bvec = b[t].astype(np.float64)[:, None] * alpha * kk
        E_pred = (alpha[:, :, None] * E
                  - np.einsum("ni,nj->nij", kk, np.einsum("nij,ni->nj", E, bvec)) + eps)
        E = w.logical(range(n)) - fp.S
        assert np.max(np.abs(E - E_pred)) <= 1e-12 * np.abs(fp.S).max()
        eps_sum += np.linalg.norm(eps, axis=(1, 2))
    assert np.all(np.linalg.norm(E, axis=(1, 2)) <= eps_sum * (1 + 1e-9))
    assert np.all(eps_sum > 0)


@pytest.mark.parametrize("gate,dl", GATES)
def test_window_commit_and_load(oracle_mod, gate, dl):
    rng = np.random.default_rng(44)
    n, W = 3, 5
    w = oracle_mod.WindowInt8Oracle(n, DK, DV, dl, W=W)
    S0 = rng.standard_normal((n, DK, DV))
    w.load(range(n), S0)
    Z0, s0 = oracle_mod.quantize_rows(S0)
    assert np.array_equal(w.Z, Z0) and np.array_equal(w.s, s0)
    q, k, v, lam, b = make_inputs(rng, 8, n, DK, dl, DV)
    for t in range(2):
        w.step(range(n), q[t], k[t], v[t], lam[t], b[t])
    S_mid = w.logical(range(n))
    w.commit([1])
    Z1, s1 = oracle_mod.quantize_rows(S_mid[1])
    assert np.array_equal(w.Z[1], Z1) and np.array_equal(w.s[1], s1)
    assert list(w.cnt) == [2, 0, 2]
    Zb = w.Z.copy()
    w.commit([1])  # empty window: unchanged
    assert np.array_equal(w.Z, Zb)
    # slot 1 now reaches its boundary W tokens after the commit
    for t in range(2, 2 + W):
        w.step(range(n), q[t % 8], k[t % 8], v[t % 8], lam[t % 8], b[t % 8])
    assert list(w.cnt) == [(2 + W) % W, 0, (2 + W) % W]
