"""Edge cases of the C ABI on the GPU: empty batches, bad slots, alignment,
slot lifecycle (load / reset / commit / read), per-slot window phases, host
buffers, the largest window.  Everything is compared with the CPU oracle."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _mods():
    import oracle
    import _harness as H
    from recurrent_state_quantization_gb300 import StatePool, LsError
    from recurrent_state_quantization_gb300 import workloads as wl
    from recurrent_state_quantization_gb300 import _native as N
    return oracle, H, StatePool, LsError, wl, N


def _inputs(w, t, dev, B=None):
    from recurrent_state_quantization_gb300 import workloads as wl
    return wl.step_inputs(w, t, device=dev)


@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 4), ("int8", 4)])
def test_empty_batch_is_noop(variant, window):
    _, _, StatePool, _, _, _ = _mods()
    pool = StatePool(3, 2, variant, "scalar", window)
    z = lambda *s: torch.empty(*s, device="cuda")
    y = pool.decode_step(torch.empty(0, dtype=torch.int32, device="cuda"), z(0, 2, D), z(0, 2, D),
                         z(0, 2, D), z(0, 2), z(0, 2))
    assert y.shape == (0, 2, D)
    assert torch.all(pool.read(range(3)) == 0)
    pool.window_commit([])
    pool.reset([])
    assert pool.status() == 0


@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 4), ("int8", 4)])
def test_out_of_range_slot_is_flagged_and_skipped(variant, window):
    oracle, H, StatePool, _, wl, N = _mods()
    w = wl.custom(batch=3, heads=2, num_slots=4, seed=5)
    pool = StatePool(4, 2, variant, "scalar", window)
    orc = H.make_oracle(variant, 8, 1, window)
    slots = torch.tensor([2, 9, 0], dtype=torch.int32, device="cuda")
    q, k, v, lam, beta = _inputs(w, 0, "cuda")
    y = pool.decode_step(slots, q, k, v, lam, beta)
    st = pool.status()
    assert st & N.LS_DEV_SLOT_RANGE
    assert torch.all(torch.isnan(y[1]))
    rows = np.array([0, 1, 4, 5])
    hq = H.host_inputs((q, k, v, lam, beta), w, rows)
    yo = orc.step(np.array([4, 5, 0, 1]), *hq)
    yg = y.reshape(6, D)[torch.as_tensor(rows, device="cuda")].double().cpu().numpy()
    assert H.relmax(yg, yo) <= 1e-4
    assert pool.status() == 0  # cleared by the previous read


@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 2), ("int8", 2)])
def test_check_slots_passes_distinct_lists(variant, window):
    """LS_CHECK_SLOTS: with distinct slot lists every state-changing call runs
    unflagged, and the outputs and states equal an unchecked pool's bit for
    bit (the check only counts slots)."""
    _, _, StatePool, _, wl, _ = _mods()
    w = wl.custom(batch=3, heads=2, num_slots=4, seed=6)
    a = StatePool(4, 2, variant, "scalar", window, check_slots=True)
    b = StatePool(4, 2, variant, "scalar", window)
    slots = torch.tensor([3, 0, 2], dtype=torch.int32, device="cuda")
    init = torch.randn(1, 2, D, D, device="cuda", generator=torch.Generator("cuda").manual_seed(4))
    for p in (a, b):
        p.load([1], init)
    for t in range(5):
        ins = _inputs(w, t, "cuda")
        ya, yb = a.decode_step(slots, *ins), b.decode_step(slots, *ins)
        assert torch.equal(ya, yb), t
    for p in (a, b):
        p.window_commit([0, 2])
        p.reset([3])
        if variant != "eager":
            p.decode_step_split_static(slots, *_inputs(w, 5, "cuda"))
    assert torch.equal(a.read(range(4)), b.read(range(4)))
    assert a.status() == 0 and b.status() == 0


def test_check_slots_flags_a_repeated_slot():
    """LS_CHECK_SLOTS: a slot named twice in one call sets LS_DEV_SLOT_DUP;
    the counts are cleared, so the next distinct list is not flagged.  Only
    calls whose repeated writes are harmless run here: the eager step (two
    warps update one dense state) and reset (two CTAs write the same zeros)."""
    _, _, StatePool, _, wl, N = _mods()
    w = wl.custom(batch=3, heads=2, num_slots=4, seed=7)
    ins = _inputs(w, 0, "cuda")
    pool = StatePool(4, 2, "eager", "scalar", 0, check_slots=True)
    pool.decode_step(torch.tensor([1, 2, 1], dtype=torch.int32, device="cuda"), *ins)
    assert pool.status() == N.LS_DEV_SLOT_DUP
    pool.decode_step(torch.tensor([1, 2, 3], dtype=torch.int32, device="cuda"), *ins)
    assert pool.status() == 0
    for variant, window in (("eager", 0), ("deferred", 2), ("int8", 2)):
        p = StatePool(4, 2, variant, "scalar", window, check_slots=True)
        p.reset([0, 3, 0])
        assert p.status() == N.LS_DEV_SLOT_DUP
        p.reset([0, 3])
        assert p.status() == 0
    # an out-of-range slot is not counted; the reset flags it itself
    p = StatePool(4, 2, "deferred", "scalar", 2, check_slots=True)
    p.reset([2, 7])
    assert p.status() == N.LS_DEV_SLOT_RANGE


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 3), ("int8", 3)])
def test_nan_input_stays_in_its_head(gate, variant, window):
    """Non-finite inputs are not checked, but their effect stays in the head
    that received them: with a NaN in one head's v, every other (request,
    head) gives bit-identical outputs and states to a run with finite inputs,
    across window ends (the per-CTA merge and the tensor-core fold process
    heads that share shared memory or a queue with the poisoned one)."""
    _, _, StatePool, _, wl, _ = _mods()
    w = wl.custom(gate=gate, batch=3, heads=2, num_slots=4, seed=9)
    a = StatePool(4, 2, variant, gate, window)
    b = StatePool(4, 2, variant, gate, window)
    slots = torch.tensor([3, 1, 0], dtype=torch.int32, device="cuda")
    keep = torch.ones(3, 2, dtype=torch.bool, device="cuda")
    keep[1, 0] = False  # request 1 (slot 1), head 0
    for t in range(8):
        q, k, v, lam, beta = _inputs(w, t, "cuda")
        ya = a.decode_step(slots, q, k, v, lam, beta)
        if t == 1:
            v = v.clone()
            v[1, 0, 5] = float("nan")
        yb = b.decode_step(slots, q, k, v, lam, beta)
        assert torch.equal(ya[keep], yb[keep]), t
        if t == 1:
            assert torch.isnan(yb[1, 0, 5])
    sa, sb = a.read(range(4)), b.read(range(4))
    for slot in (0, 2, 3):
        assert torch.equal(sa[slot], sb[slot])
    assert torch.equal(sa[1, 1], sb[1, 1])
    assert a.status() == 0 and b.status() == 0


def test_argument_errors():
    _, _, StatePool, LsError, wl, N = _mods()
    pool = StatePool(2, 2, "eager", "scalar", 0)
    w = wl.custom(batch=2, heads=2, num_slots=2, seed=3)
    q, k, v, lam, beta = _inputs(w, 0, "cuda")
    slots = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    buf = torch.empty(2 * 2 * D + 1, device="cuda")
    q_bad = buf[1:].view(2, 2, D)  # 4-byte offset: not 16-byte aligned
    q_bad.copy_(q)
    with pytest.raises(LsError) as e:
        pool.decode_step(slots, q_bad, k, v, lam, beta)
    assert e.value.code == N.LS_ERR_ALIGN
    w3 = wl.custom(batch=3, heads=2, num_slots=3, seed=3)
    with pytest.raises(LsError) as e:
        pool.decode_step(torch.tensor([0, 1, 0], dtype=torch.int32, device="cuda"),
                         *_inputs(w3, 0, "cuda"))
    assert e.value.code == N.LS_ERR_SLOT
    with pytest.raises(LsError) as e:
        StatePool(2, 2, "int8", "scalar", 0)  # window 0 is not a window
    assert e.value.code == N.LS_ERR_SIZE
    with pytest.raises(LsError) as e:
        StatePool(2, 2, "deferred", "scalar", 257)
    assert e.value.code == N.LS_ERR_SIZE


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 5), ("int8", 5)])
def test_beta_zero_no_decay_keeps_state(gate, variant, window):
    oracle, H, StatePool, _, wl, _ = _mods()
    w = wl.custom(gate=gate, batch=2, heads=3, num_slots=2, seed=8)
    pool = StatePool(2, 3, variant, gate, window)
    S0 = wl.initial_state(w, "cuda")
    pool.load(range(2), S0)
    before = pool.read(range(2))
    for t in range(7):
        q, k, v, lam, beta = _inputs(w, t, "cuda")
        y = pool.decode_step(range(2), q, k, v, torch.zeros_like(lam), torch.zeros_like(beta))
        expect = torch.einsum("bhij,bhi->bhj", before.double(), q.double())
        assert H.relmax(y.double().cpu().numpy(), expect.cpu().numpy()) <= 1e-5
    after = pool.read(range(2))
    if variant == "eager":
        assert torch.equal(after, before)
    else:
        assert H.relmax(after.double().cpu().numpy(), before.double().cpu().numpy()) <= 1e-6


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant", ["eager", "deferred", "int8"])
def test_load_then_read(gate, variant):
    oracle, H, StatePool, _, wl, _ = _mods()
    w = wl.custom(gate=gate, batch=3, heads=2, num_slots=5, seed=9)
    pool = StatePool(5, 2, variant, gate, 4 if variant != "eager" else 0)
    S = wl.initial_state(w, "cuda", scale=3.0)[:3].contiguous()
    S[1, 0, 7, :] = 0.0  # a zero key row
    slots = torch.tensor([4, 0, 2], dtype=torch.int32, device="cuda")
    pool.load(slots, S)
    back = pool.read(slots)
    if variant != "int8":
        assert torch.equal(back, S)
    else:
        Z, s = pool.read_int8(slots)
        Zo, so = oracle.quantize_rows(S.double().cpu().numpy())
        assert np.array_equal(Z.cpu().numpy(), Zo)
        assert np.array_equal(s.cpu().numpy(), so)
        deq = oracle.dequantize_rows(Zo, so)
        assert H.relmax(back.double().cpu().numpy(), deq) <= 1e-7
    untouched = pool.read([1, 3])
    assert torch.all(untouched == 0)


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window", [("deferred", 8), ("int8", 8)])
def test_commit_mid_window_and_reset(gate, variant, window):
    oracle, H, StatePool, _, wl, _ = _mods()
    w = wl.custom(gate=gate, batch=4, heads=2, num_slots=4, seed=12, lam_scale=0.3)
    p = H.Pair(w, variant, window)
    for t in range(5):
        p.step(t)
    before = p.pool.read(p.slot_idx).double().cpu().numpy()
    commit_slots = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    p.pool.window_commit(commit_slots)
    st_idx = np.concatenate([np.arange(2) + 2 * 1, np.arange(2) + 2 * 3])
    p.orc.commit(st_idx)
    ln, lb = p.pool.read_log_meta(torch.arange(4, dtype=torch.int32, device="cuda"))
    assert ln.cpu().tolist() == [[5, 5], [0, 0], [5, 5], [0, 0]]
    assert torch.all(lb[[1, 3]] == 0)
    after = p.pool.read(p.slot_idx).double().cpu().numpy()
    if variant == "deferred":
        assert H.relmax(after, before) <= 1e-6
    else:
        frac, mx = p.code_mismatch()
        assert mx <= 1 and frac <= 1e-4
        assert H.rel_l2(after, before) <= 1e-2
    p.pool.window_commit(commit_slots)  # empty logs: unchanged
    assert np.array_equal(p.pool.read(p.slot_idx).double().cpu().numpy(), after)
    for t in range(5, 5 + window):  # windows now end at different tokens per slot
        p.step(t)
    check = p.y_rel_l2() if variant == "int8" else p.y_err()
    assert check <= (2e-3 if variant == "int8" else 1e-4)
    p.pool.reset(commit_slots)
    z = p.pool.read(commit_slots)
    assert torch.all(z == 0)
    ln, _ = p.pool.read_log_meta(commit_slots)
    assert torch.all(ln == 0)
    assert p.pool.status() == 0


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window,fmt", [("eager", 0, {}), ("deferred", 4, {}), ("int8", 4, {}),
                                                ("int8", 5, {"r16": True}),
                                                ("int8", 4, {"col_scales": True})])
def test_changing_batches_keep_per_slot_phase(gate, variant, window, fmt):
    """Different subsets of slots decode at different tokens (continuous
    batching), so every slot is at its own position in its window and the
    window-end queue holds a different subset of states at every token
    (per-row INT8 scales); the column-scale format folds in the step kernel."""
    oracle, H, StatePool, _, wl, _ = _mods()
    P, Hh = 6, 2
    w = wl.custom(gate=gate, batch=P, heads=Hh, num_slots=P, seed=21, lam_scale=0.3)
    pool = StatePool(P, Hh, variant, gate, window, **fmt)
    orc = H.make_oracle(variant, P * Hh, w.dl, window, **fmt)
    rng = np.random.default_rng(0)
    worst = 0.0
    for t in range(23):
        nb = int(rng.integers(1, P + 1))
        slots = np.sort(rng.choice(P, nb, replace=False)).astype(np.int32)
        q, k, v, lam, beta = _inputs(w, t, "cuda")
        sel = torch.as_tensor(np.arange(nb), device="cuda")
        ins = [x[:nb].contiguous() for x in (q, k, v, lam, beta)]
        y = pool.decode_step(torch.as_tensor(slots, device="cuda"), *ins)
        sub = wl.custom(gate=gate, batch=nb, heads=Hh, num_slots=P, seed=21)
        rows = np.arange(nb * Hh)
        yo = orc.step((slots[:, None] * Hh + np.arange(Hh)).reshape(-1),
                      *H.host_inputs(ins, sub, rows))
        yg = y.reshape(-1, D).double().cpu().numpy()
        worst = max(worst, H.rel_l2(yg, yo) if variant == "int8" else H.relmax(yg, yo))
    assert worst <= (2e-3 if variant == "int8" else 1e-4)
    S = pool.read(range(P)).reshape(-1, D, D).double().cpu().numpy()
    So = orc.logical(np.arange(P * Hh))
    if variant == "int8":
        assert H.rel_l2(S, So) <= 2e-3
    else:
        assert H.relmax(S, So) <= 1e-4
    if variant != "eager":
        ln, _ = pool.read_log_meta(range(P))
        cnt = orc.cnt if variant == "int8" else orc.L
        assert np.array_equal(ln.cpu().numpy().reshape(-1), cnt)


@pytest.mark.parametrize("variant,window", [("eager", 0), ("deferred", 4), ("int8", 4)])
def test_host_buffer_entry_point(variant, window):
    _, H, StatePool, _, wl, _ = _mods()
    w = wl.custom(gate="per_key", batch=3, heads=2, num_slots=3, seed=4)
    a = StatePool(3, 2, variant, "per_key", window)
    b = StatePool(3, 2, variant, "per_key", window)
    slots = torch.tensor([2, 0, 1], dtype=torch.int32)
    for t in range(6):
        ins = _inputs(w, t, "cuda")
        ya = a.decode_step(slots.cuda(), *ins)
        hs = [x.cpu().pin_memory() for x in ins]
        yb = torch.empty(3, 2, D).pin_memory()
        b.decode_step_host(slots.pin_memory(), *hs, yb)
        torch.cuda.synchronize()
        assert torch.equal(ya.cpu(), yb)
    assert torch.equal(a.read(range(3)), b.read(range(3)))


@pytest.mark.parametrize("variant", ["deferred", "int8"])
def test_largest_window(variant):
    oracle, H, StatePool, _, wl, _ = _mods()
    w = wl.custom(gate="scalar", batch=2, heads=2, num_slots=2, tokens=260, seed=30,
                  lam_scale=0.02)
    p = H.Pair(w, variant, 256)
    for t in range(w.tokens):
        if variant == "int8" and t == 256:
            p.force_boundary()
        p.step(t)
        if variant == "int8" and t == 255:
            frac, mx = p.code_mismatch()
            assert mx <= 1 and frac <= 1e-4
    ln, _ = p.pool.read_log_meta(p.slot_idx)
    assert torch.all(ln == 4)
    if variant == "int8":
        assert p.y_rel_l2() <= 2e-3
    else:
        assert p.y_err() <= 1e-4 and p.state_err() <= 1e-4


@pytest.mark.parametrize("gate", ["scalar", "per_key"])
@pytest.mark.parametrize("variant,window,fmt", [("deferred", 4, {}), ("int8", 4, {}),
                                                ("int8", 3, {"r16": True}),
                                                ("int8", 4, {"col_scales": True}),
                                                ("int8", 5, {"compensators": 2})])
def test_lifecycle_fuzz(gate, variant, window, fmt):
    """Seeded random interleaving of decode calls on random slot subsets with
    resets, loads and window commits of random slots: every slot has its own
    window phase, the window-end queue (per-row INT8 scales) sees a different
    subset at every call, and the lifecycle calls run between folds.  Each
    call's outputs, the final logical states and the log lengths are compared
    with the oracle driven through the same operations."""
    oracle, H, StatePool, _, wl, _ = _mods()
    P, Hh = 6, 2
    w = wl.custom(gate=gate, batch=P, heads=Hh, num_slots=P, seed=23, lam_scale=0.3)
    pool = StatePool(P, Hh, variant, gate, window, **fmt)
    orc = H.make_oracle(variant, P * Hh, w.dl, window, **fmt)
    rng = np.random.default_rng(7)
    g = torch.Generator(device="cpu").manual_seed(3)
    sidx = lambda s: (s[:, None] * Hh + np.arange(Hh)).reshape(-1)
    worst, t = 0.0, 0
    for op in range(48):
        kind = rng.choice(["step"] * 6 + ["reset", "load", "commit"])
        if kind == "step":
            nb = int(rng.integers(1, P + 1))
            slots = np.sort(rng.choice(P, nb, replace=False)).astype(np.int32)
            ins = [x[:nb].contiguous() for x in _inputs(w, t, "cuda")]
            t += 1
            y = pool.decode_step(torch.as_tensor(slots, device="cuda"), *ins)
            sub = wl.custom(gate=gate, batch=nb, heads=Hh, num_slots=P, seed=23)
            yo = orc.step(sidx(slots), *H.host_inputs(ins, sub, np.arange(nb * Hh)))
            yg = y.reshape(-1, D).double().cpu().numpy()
            worst = max(worst, H.rel_l2(yg, yo) if variant == "int8" else H.relmax(yg, yo))
            continue
        n = int(rng.integers(1, 3))
        slots = np.sort(rng.choice(P, n, replace=False)).astype(np.int32)
        st = torch.as_tensor(slots, device="cuda")
        if kind == "reset":
            pool.reset(st)
            orc.reset(sidx(slots))
        elif kind == "load":
            S = (torch.randn(n, Hh, D, D, generator=g) * 0.5).float()
            pool.load(st, S.to("cuda"))
            orc.load(sidx(slots), S.double().numpy().reshape(-1, D, D))
        else:
            pool.window_commit(st)
            orc.commit(sidx(slots))
    assert t > 0
    assert worst <= (2e-3 if variant == "int8" else 1e-4), worst
    S = pool.read(range(P)).reshape(-1, D, D).double().cpu().numpy()
    So = orc.logical(np.arange(P * Hh))
    if variant == "int8":
        assert H.rel_l2(S, So) <= 2e-3
    else:
        assert H.relmax(S, So) <= 1e-4
    ln, _ = pool.read_log_meta(range(P))
    # compensator pools: the log holds the r pairs ahead of the window's tokens
    cnt = orc.cnt + fmt.get("compensators", 0) if variant == "int8" else orc.L
    assert np.array_equal(ln.cpu().numpy().reshape(-1), cnt)
    assert pool.status() == 0
