"""Parity of the CUDA decode step (through the C ABI) with the CPU oracle.

Bars (the tolerance stated for this path):
  eager / deferred FP32: max relative error <= 1e-4 on y and on the logical
      state S (per head: max |gpu - oracle| / max |oracle|);
  per-window INT8: codes differ by at most 1 LSB on at most 1e-4 of the
      elements at every window boundary, and y within 2e-3 relative L2.
Small cases compare every head at every token; the full-size workloads run the
whole batch on the GPU in the launch configuration the benchmark times and
compare a seeded sample of heads with the oracle.

INT8 trajectories are compared one window at a time: a legitimate one-LSB
code flip at a rounding boundary (FP32 kernel vs double oracle) perturbs every
later window, so two free-running quantized trajectories drift apart.  At each
window start the oracle's own state is rounded to FP32 and loaded into both
sides (no GPU value enters the oracle).  The free-running divergence is
measured separately as drift (test_int8_free_running_drift).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-4
Y_L2_TOL = 2e-3
CODE_FRAC_TOL = 1e-4
# compensator pools: the fitted pairs carry the FP32 rounding of the state's
# dominant component (~2^-22 sigma_1, times sigma_1 / sigma_r through the
# deflations) into a residual whose step is ~max|R| / 127, so near-tie flips
# are ~10x more frequent than in the plain format
CODE_FRAC_TOL_COMP = 2e-3
# ... the pairs themselves: pair h inherits the FP32 rounding of the earlier
# pairs amplified by sigma_1 / sigma_h through the deflations (up to ~1e3 on
# these states); the residual's factors (absmax of a row or column of a
# residual ~10x smaller than the state) inherit that difference relatively
COMP_TOL = 1e-3
FACTOR_TOL_COMP = 1e-2
# FP16 records (LeapQuant §4.1, §4.3): a record element whose FP32 (kernel)
# and fp64 (oracle) values straddle a binary16 rounding boundary is stored
# one binary16 step (2^-11 relative) apart on the two sides, with
# probability ~ their difference / 2^-11 (~1e-4 per element).  That moves S
# by one step of the record's k_i u_j in one row or column: a row's absmax
# by at most 2^-10 relative (k and u of one record), the codes of that row
# or column by up to 127 * 2^-10 ~ 0.12 LSB, so near-tie flips there are
# ~10x more frequent than in the FP32-record format; stored pairs differ by
# one binary16 step in each factor.
FACTOR_TOL_R16 = 2.0 ** -10
CODE_FRAC_TOL_R16 = 2e-3
# binary16 pairs: pair elements may sit one binary16 step apart (2^-11
# relative in k~ and in u~); every later pair is fitted, by three power
# steps that do not converge, to a residual that differs by those steps, so
# it can turn within a near-degenerate singular subspace.  The pairs'
# products are checked loosely; the boundary states are checked tightly
# (boundary_step_err).
COMP_TOL_R16_PAIRS = 5e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _harness():
    import _harness as H  # noqa: WPS433 (tests dir is on sys.path)
    return H


def check_fp32(p, where=""):
    ye, se = p.y_err(), p.state_err()
    assert ye <= FP32_TOL, f"{where} y max rel err {ye:.3g}"
    assert se <= FP32_TOL, f"{where} state max rel err {se:.3g}"
    return ye, se


# key-row / column factors at a window end are functions (absmax, row mean)
# of each side's own end-of-window state, which agree within the FP32
# tolerance; at a restart both sides quantize the same FP32 state
FACTOR_TOL = FP32_TOL


def run_lockstep(p, tokens, pool_id=0, code_checks=None):
    """Step every token; for INT8 restart each window from the oracle's state
    on both sides and check the codes at its end."""
    for t in range(tokens):
        if p.variant == "int8" and t % p.window == 0 and t > 0:
            p.force_boundary()
        p.step(t, pool_id=pool_id)
        if p.variant == "int8" and (t + 1) % p.window == 0 and p.r16 and p.compensators:
            # binary16 pairs: a pair element whose FP32 and fp64 fits straddle
            # a binary16 rounding boundary is stored one step apart, and the
            # residual (quantized against a ~10-100x smaller row maximum)
            # absorbs that step, so codes are not comparable one to one; each
            # side's boundary state is still within half a code step of the
            # same unquantized state
            be = p.boundary_step_err()
            assert be <= 1.0, f"token {t}: boundary states differ by {be:.3g} x the bound"
            ce = p.comp_err()
            assert ce <= COMP_TOL_R16_PAIRS, f"token {t}: compensator pairs rel err {ce:.3g}"
        elif p.variant == "int8" and (t + 1) % p.window == 0:
            frac, mx = p.code_mismatch()
            if code_checks is not None:
                code_checks.append((t, frac, mx))
            assert mx <= 1, f"token {t}: codes differ by {mx} LSB"
            tol = (CODE_FRAC_TOL_COMP if p.compensators else
                   CODE_FRAC_TOL_R16 if p.r16 else CODE_FRAC_TOL)
            assert frac <= tol, f"token {t}: {frac:.3g} of codes differ"
            fe = p.factor_err()
            ftol = (FACTOR_TOL_COMP if p.compensators else
                    FACTOR_TOL_R16 if p.r16 else FACTOR_TOL)
            assert fe <= ftol, f"token {t}: scale / smoothing factors rel err {fe:.3g}"
            if p.compensators:
                ce = p.comp_err()
                assert ce <= COMP_TOL, f"token {t}: compensator pairs rel err {ce:.3g}"


def check_int8(p):
    l2 = p.y_rel_l2()
    assert l2 <= Y_L2_TOL, f"y rel L2 {l2:.3g}"
    return l2


# ---------------------------------------------------------------------------
# the smallest workload, every head, every token
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 16), ("int8", 16)])
def test_gdn_b1_h4_t64(variant, window):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[0]
    p = H.Pair(w, variant, window)
    run_lockstep(p, w.tokens)
    if variant == "int8":
        check_int8(p)
    else:
        check_fp32(p)
    assert p.pool.status() == 0


# ---------------------------------------------------------------------------
# ragged small cases: permuted slots, unused slots, windows that do not divide T
# ---------------------------------------------------------------------------

CASES = [("eager", 0), ("deferred", 1), ("deferred", 3), ("deferred", 16),
         ("int8", 1), ("int8", 3), ("int8", 16), ("int8", 40)]

# the plain update rule (no delta-rule correction): RWKV6 with the per-key gate


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 1), ("deferred", 4),
                                            ("deferred", 16)])
def test_small_ragged_plain(gate, variant, window):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.custom("ragged-plain", gate=gate, batch=5, heads=3, tokens=37, num_slots=7,
                  windows=(max(window, 1),), merge_interval=max(window, 1), permute_slots=True,
                  seed=31 + window, lam_scale=0.3)
    p = H.Pair(w, variant, window, plain=True)
    run_lockstep(p, w.tokens)
    check_fp32(p)
    assert p.pool.status() == 0


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window,cols,comp", [c + (False, 0) for c in CASES] +
                         [("int8", 1, True, 0), ("int8", 3, True, 0), ("int8", 16, True, 0),
                          ("int8", 1, False, 2), ("int8", 5, False, 4), ("int8", 16, True, 4)])
def test_small_ragged(gate, variant, window, cols, comp):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.custom("ragged", gate=gate, batch=5, heads=3, tokens=37, num_slots=7,
                  windows=(max(window, 1),), merge_interval=max(window, 1), permute_slots=True,
                  seed=11 + window, lam_scale=0.3)
    p = H.Pair(w, variant, window, col_scales=cols, compensators=comp)
    run_lockstep(p, w.tokens)
    if variant == "int8":
        check_int8(p)
    else:
        check_fp32(p)
    if variant != "eager":
        ln, _ = p.pool.read_log_meta(p.slot_idx)
        assert torch.all(ln == comp + (w.tokens % max(window, 1)))
    assert p.pool.status() == 0


# ---------------------------------------------------------------------------
# full-size workloads, sampled heads
# ---------------------------------------------------------------------------

def _full(wi, variant, window, n_sample, tokens=None, pools=1, prewarm=None, cols=False, comp=0):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[wi]
    T = w.tokens if tokens is None else tokens
    results = []
    for pool_id in range(pools):
        p = H.Pair(w, variant, window, n_sample=n_sample, seed=pool_id, col_scales=cols,
                   compensators=comp)
        if prewarm is not None:
            prewarm(p, pool_id)
        checks = []
        for t in range(T):
            if variant == "int8" and t % window == 0 and t > 0:
                p.force_boundary()
            p.step(t, pool_id=pool_id)
            if variant == "int8" and (t + 1) % window == 0:
                frac, mx = p.code_mismatch()
                checks.append((t, frac, mx))
                assert p.factor_err() <= (FACTOR_TOL_COMP if comp else FACTOR_TOL), t
                if comp:
                    assert p.comp_err() <= COMP_TOL, t
        results.append((p, checks))
    return results


def _assert_full(results, variant):
    for p, checks in results:
        if variant == "int8":
            check_int8(p)
            for t, frac, mx in checks:
                tol = CODE_FRAC_TOL_COMP if p.compensators else CODE_FRAC_TOL
                assert mx <= 1 and frac <= tol, (t, frac, mx)
        else:
            check_fp32(p)
        assert p.pool.status() == 0


@pytest.mark.parametrize("variant,window", [("eager", 0), ("int8", 64)])
def test_gdn_pool_b64_h48_t1024_outliers(variant, window):
    _assert_full(_full(1, variant, window, n_sample=24), variant)


@pytest.mark.parametrize("variant,window,cols,comp", [("eager", 0, False, 0), ("deferred", 16, False, 0),
                                                      ("int8", 32, False, 0), ("int8", 32, True, 0),
                                                      ("int8", 32, True, 4)])
def test_kda_b128_h32_t512_longlived(variant, window, cols, comp):
    _assert_full(_full(2, variant, window, n_sample=16, cols=cols, comp=comp), variant)


def _prewarm_factory(tokens):
    """Warm the sampled states by `tokens` eager updates on both sides
    independently (GPU: eager kernel then ls_pool_load; oracle: its own eager
    recurrence), so that no oracle input comes from the GPU."""
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()

    def prewarm(p, pool_id):
        w = p.w
        eager = StatePool(w.num_slots, w.heads, "eager", w.gate, 0, device=p.dev)
        orc = H.make_oracle("eager", w.num_slots * w.heads, w.dl, 0)
        for t in range(-tokens, 0):
            inputs = wl.step_inputs(w, t, pool=pool_id, device=p.dev, masks=p.masks)
            eager.decode_step(p.slot_idx, *inputs)
            orc.step(p.sample.state_idx, *H.host_inputs(inputs, w, p.sample.rows))
        all_slots = torch.arange(w.num_slots, dtype=torch.int32, device=p.dev)
        p.pool.load(all_slots, eager.read(all_slots))
        p.orc.load(p.sample.state_idx, orc.logical(p.sample.state_idx))
    return prewarm


@pytest.mark.parametrize("variant,window,cols", [("eager", 0, False), ("deferred", 16, False),
                                                 ("int8", 8, False), ("int8", 16, False),
                                                 ("int8", 32, False), ("int8", 64, False),
                                                 ("int8", 128, False), ("int8", 16, True)])
def test_gdn_serving_b256_h48_4pools(variant, window, cols):
    from recurrent_state_quantization_gb300 import workloads as wl
    w = wl.WORKLOADS[3]
    _assert_full(_full(3, variant, window, n_sample=6, pools=w.pools, cols=cols,
                       prewarm=_prewarm_factory(w.prewarm_tokens)), variant)


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window,cols", [("deferred", 1, False), ("deferred", 5, False),
                                                 ("deferred", 16, False), ("int8", 1, False),
                                                 ("int8", 5, False), ("int8", 16, True)])
def test_small_ragged_bf16_keys(gate, variant, window, cols):
    """bfloat16 key-side log factors (DeltaLog §3.4) against the oracle's."""
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.custom("ragged-k16", gate=gate, batch=5, heads=3, tokens=37, num_slots=7,
                  windows=(window,), merge_interval=window, permute_slots=True,
                  seed=51 + window, lam_scale=0.3)
    p = H.Pair(w, variant, window, col_scales=cols, k16=True)
    run_lockstep(p, w.tokens)
    if variant == "int8":
        check_int8(p)
    else:
        check_fp32(p)
    assert p.pool.status() == 0


@pytest.mark.parametrize("variant,window", [("deferred", 16), ("int8", 16)])
def test_gdn_serving_b256_h48_bf16_keys(variant, window):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[3]
    p = H.Pair(w, variant, window, n_sample=6, k16=True)
    _prewarm_factory(w.prewarm_tokens)(p, 0)
    run_lockstep(p, 64)
    if variant == "int8":
        check_int8(p)
    else:
        check_fp32(p)
    assert p.pool.status() == 0


# ---------------------------------------------------------------------------
# FP16 records (LeapQuant §4.1, §4.3): k, u and the compensator pairs in binary16
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("window,cols,comp", [(1, False, 0), (5, False, 0), (16, False, 0),
                                              (40, False, 0), (16, True, 0), (5, False, 2),
                                              (16, True, 4)])
def test_small_ragged_fp16_records(gate, window, cols, comp):
    """The INT8 window with binary16 records against the oracle's: the row-scale
    format folds on the tensor cores, the others in the step kernel."""
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.custom("ragged-r16", gate=gate, batch=5, heads=3, tokens=37, num_slots=7,
                  windows=(window,), merge_interval=window, permute_slots=True,
                  seed=61 + window, lam_scale=0.3)
    p = H.Pair(w, "int8", window, col_scales=cols, compensators=comp, r16=True)
    run_lockstep(p, w.tokens)
    check_int8(p)
    assert p.pool.status() == 0
    ln, _ = p.pool.read_log_meta(p.slot_idx)
    assert torch.all(ln == comp + (w.tokens % window))


def test_gdn_serving_b256_h48_fp16_records():
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[3]
    p = H.Pair(w, "int8", 16, n_sample=6, r16=True)
    _prewarm_factory(w.prewarm_tokens)(p, 0)
    run_lockstep(p, 64)
    check_int8(p)
    assert p.pool.status() == 0


# ---------------------------------------------------------------------------
# split replay (DeltaLog §5.3): the coefficients from a prepare kernel
# ---------------------------------------------------------------------------

SPLIT_CASES = [("deferred", 1, {}), ("deferred", 5, {}), ("deferred", 16, {}),
               ("deferred", 7, {"plain": True}), ("deferred", 6, {"k16": True}),
               ("int8", 1, {}), ("int8", 5, {}), ("int8", 16, {"col_scales": True}),
               ("int8", 6, {"col_scales": True, "compensators": 2}), ("int8", 13, {"k16": True}),
               ("int8", 9, {"r16": True}), ("int8", 6, {"r16": True, "compensators": 2})]


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window,fmt", SPLIT_CASES)
def test_small_ragged_split(gate, variant, window, fmt):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.custom("ragged-split", gate=gate, batch=5, heads=3, tokens=37, num_slots=7,
                  windows=(window,), merge_interval=window, permute_slots=True,
                  seed=71 + window, lam_scale=0.3)
    p = H.Pair(w, variant, window, split=True, **fmt)
    run_lockstep(p, w.tokens)
    if variant == "int8":
        check_int8(p)
    else:
        check_fp32(p)
    assert p.pool.status() == 0


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window,fmt", SPLIT_CASES)
def test_split_equals_fused_bitwise(gate, variant, window, fmt):
    """The prepare kernel reduces each coefficient exactly as the fused replay
    does, so the two entry points leave the same bits in y and in the pool."""
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import workloads as wl
    dev = torch.device("cuda")
    w = wl.custom("split-bits", gate=gate, batch=6, heads=5, tokens=3 * window + 4, num_slots=9,
                  windows=(window,), merge_interval=window, permute_slots=True, seed=91)
    fused = StatePool(w.num_slots, w.heads, variant, gate, window, device=dev, **fmt)
    split = StatePool(w.num_slots, w.heads, variant, gate, window, device=dev, **fmt)
    slots = wl.slot_index(w, dev)
    all_slots = torch.arange(w.num_slots, dtype=torch.int32, device=dev)
    g = torch.Generator(device="cpu").manual_seed(5)
    S0 = torch.randn(w.num_slots, w.heads, 128, 128, generator=g).to(dev) * 0.3
    fused.load(all_slots, S0)
    split.load(all_slots, S0)
    masks = wl.static_masks(w, dev)
    for t in range(w.tokens):
        ins = wl.step_inputs(w, t, device=dev, masks=masks)
        yf = fused.decode_step(slots, *ins)
        ys = split.decode_step_split(slots, *ins)
        assert torch.equal(yf, ys), f"token {t}: y differs"
    assert torch.equal(fused.read(all_slots), split.read(all_slots))
    if variant == "int8":
        cf, sf = fused.read_int8(all_slots)
        cs, ss = split.read_int8(all_slots)
        assert torch.equal(cf, cs) and torch.equal(sf, ss)
    assert fused.status() == 0 and split.status() == 0


@pytest.mark.parametrize("variant,window", [("deferred", 8), ("int8", 16)])
def test_gdn_serving_b256_h48_split(variant, window):
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[3]
    p = H.Pair(w, variant, window, n_sample=6, split=True)
    _prewarm_factory(w.prewarm_tokens)(p, 0)
    run_lockstep(p, 48)
    if variant == "int8":
        check_int8(p)
    else:
        check_fp32(p)
    assert p.pool.status() == 0


def test_split_scratch_bytes_and_errors():
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import _native as N
    dev = torch.device("cuda")
    for variant, W, comp, expect_cap in (("deferred", 16, 0, 18), ("int8", 5, 0, 6),
                                         ("int8", 16, 4, 24), ("int8", 1, 0, 6)):
        pool = StatePool(4, 3, variant, "scalar", W, device=dev, compensators=comp,
                         col_scales=comp > 0)
        assert pool.split_scratch_bytes(4) == 4 * 3 * expect_cap * 8
        assert pool.split_scratch_bytes(0) == 0
        slots = torch.arange(4, dtype=torch.int32, device=dev)
        q = torch.zeros(4, 3, 128, device=dev)
        lam = torch.zeros(4, 3, device=dev)
        short = torch.empty(pool.split_scratch_bytes(4) - 16, dtype=torch.uint8, device=dev)
        with pytest.raises(RuntimeError, match="buffer too small"):
            pool.decode_step_split(slots, q, q, q, lam, lam, scratch=short)
    eager = StatePool(4, 3, "eager", "scalar", 0, device=dev)
    with pytest.raises(RuntimeError, match="invalid"):
        eager.split_scratch_bytes(4)
    assert N.LS_ABI_VERSION == 5


@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 16)])
def test_rwkv6_b128_h32_t512(variant, window):
    """RWKV6 (per-key decay, raw (k, v) updates) on the KDA 128x32 shapes."""
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[2]
    p = H.Pair(w, variant, window, n_sample=16, plain=True)
    run_lockstep(p, w.tokens)
    check_fp32(p)
    assert p.pool.status() == 0


def test_gdn_serving_b256_h48_compensators():
    """The full LeapQuant boundary format (4 compensator pairs + smoothed
    per-value-column INT8) on one 256x48 serving pool, W = 16."""
    from recurrent_state_quantization_gb300 import workloads as wl
    w = wl.WORKLOADS[3]
    _assert_full(_full(3, "int8", 16, n_sample=6, pools=1, cols=True, comp=4,
                       prewarm=_prewarm_factory(w.prewarm_tokens)), "int8")


@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 16), ("int8", 32)])
def test_kda_drift_b32_h32_t8192(variant, window):
    _assert_full(_full(4, variant, window, n_sample=4), variant)


# ---------------------------------------------------------------------------
# free-running INT8: the divergence between two quantized trajectories
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("wi,window,n_sample", [(1, 64, 12), (2, 32, 8), (4, 32, 4)])
def test_int8_free_running_drift(wi, window, n_sample):
    """Without restarts, rounding-boundary flips make two INT8 trajectories
    separate; over many windows the GPU and oracle INT8 trajectories become as
    different as any two quantized trajectories.  What must hold is that the
    GPU's INT8 trajectory is no further from the FP32 trajectory than the
    oracle's own INT8 trajectory is (same quantization drift).  The drift per
    1024-token block is printed."""
    from recurrent_state_quantization_gb300 import workloads as wl
    H = _harness()
    w = wl.WORKLOADS[wi]
    gi = H.Pair(w, "int8", window, n_sample=n_sample)
    fo = H.make_oracle("eager", w.num_slots * w.heads, w.dl, 0)
    acc = {"gpu_orc": 0.0, "gpu_fp": 0.0, "orc_fp": 0.0, "den": 0.0}
    block = dict(acc)
    for t in range(w.tokens):
        y, yo = gi.step(t)
        inputs = wl.step_inputs(w, t, device=gi.dev, masks=gi.masks)
        yf = fo.step(gi.sample.state_idx, *H.host_inputs(inputs, w, gi.sample.rows))
        yg = y.reshape(-1, 128)[torch.as_tensor(gi.sample.rows, device=gi.dev)]
        yg = yg.double().cpu().numpy()
        for d in (acc, block):
            d["gpu_orc"] += float(((yg - yo) ** 2).sum())
            d["gpu_fp"] += float(((yg - yf) ** 2).sum())
            d["orc_fp"] += float(((yo - yf) ** 2).sum())
            d["den"] += float((yf ** 2).sum())
        if (t + 1) % 1024 == 0 or t + 1 == w.tokens:
            b = {k_: (block[k_] / block["den"]) ** 0.5 for k_ in ("gpu_orc", "gpu_fp", "orc_fp")}
            print(f"drift {w.name} tokens <= {t + 1}: y relL2 gpu-int8 vs fp32 {b['gpu_fp']:.3g}, "
                  f"oracle-int8 vs fp32 {b['orc_fp']:.3g}, gpu-int8 vs oracle-int8 "
                  f"{b['gpu_orc']:.3g}")
            block = {k_: 0.0 for k_ in block}
    r = {k_: (acc[k_] / acc["den"]) ** 0.5 for k_ in ("gpu_orc", "gpu_fp", "orc_fp")}
    print(f"drift {w.name}: {r}")
    assert r["gpu_fp"] <= 1.25 * r["orc_fp"] + 1e-6
    S_fp = fo.logical(gi.sample.state_idx)
    print(f"drift {w.name}: final state relL2 int8-vs-fp32 gpu "
          f"{H.rel_l2(gi.pool.read(gi.slot_idx).reshape(-1, 128, 128)[torch.as_tensor(gi.sample.rows, device=gi.dev)].double().cpu().numpy(), S_fp):.3g}"
          f", oracle {H.rel_l2(gi.orc.logical(gi.sample.state_idx), S_fp):.3g}")
