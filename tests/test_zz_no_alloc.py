"""The allocation-free split-replay step (ls_decode_step_split_static, its
coefficient scratch in the library's fixed device array) against the
caller-scratch entry point (ls_decode_step_split): twin pools, two calls in a
row, the same bits in y and in the pools.  Collected last so that it also
runs after every other GPU test in the same process."""
import ctypes as C

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    """Runs alone in a fresh process as well as after the other GPU tests:
    skip without a GPU, build the library, make device 0 current."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _twins(variant, gate, window, pre, **fmt):
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import workloads as wl
    dev = torch.device("cuda")
    w = wl.custom("no-alloc", gate=gate, batch=5, heads=6, tokens=pre + 2, num_slots=8,
                  windows=(window,), merge_interval=window, permute_slots=True, seed=29)
    a = StatePool(w.num_slots, w.heads, variant, gate, window, device=dev, **fmt)
    b = StatePool(w.num_slots, w.heads, variant, gate, window, device=dev, **fmt)
    all_slots = torch.arange(w.num_slots, dtype=torch.int32, device=dev)
    g = torch.Generator(device="cpu").manual_seed(3)
    S0 = (torch.randn(w.num_slots, w.heads, 128, 128, generator=g) * 0.3).to(dev)
    a.load(all_slots, S0)
    b.load(all_slots, S0)
    slots = wl.slot_index(w, dev)
    masks = wl.static_masks(w, dev)
    ins = [wl.step_inputs(w, t, device=dev, masks=masks) for t in range(pre + 2)]
    for t in range(pre):  # live log entries before the compared calls
        a.decode_step(slots, *ins[t])
        b.decode_step(slots, *ins[t])
    return a, b, slots, ins[pre:], all_slots


@pytest.mark.parametrize("variant,gate,window,pre,fmt", [
    ("deferred", "scalar", 5, 2, {}),
    ("deferred", "per_key", 6, 3, {"k16": True}),
    ("int8", "scalar", 3, 1, {}),  # the second call closes the window
    ("int8", "per_key", 4, 2, {"col_scales": True, "compensators": 2}),
])
def test_static_scratch_matches_caller_scratch(variant, gate, window, pre, fmt):
    a, b, slots, ins, all_slots = _twins(variant, gate, window, pre, **fmt)
    for t, x in enumerate(ins):
        ya = a.decode_step_split(slots, *x)
        yb = b.decode_step_split_static(slots, *x)
        assert torch.equal(ya, yb), f"call {t}: y differs"
    assert torch.equal(a.read(all_slots), b.read(all_slots))
    if variant == "int8":
        assert all(torch.equal(u, v) for u, v in zip(a.read_int8(all_slots), b.read_int8(all_slots)))
    assert a.status() == 0 and b.status() == 0


def test_static_scratch_rejects_oversize_batch():
    """batch * H * 258 coefficient pairs of 8 bytes at the largest window
    exceed the fixed array; the call returns LS_ERR_SIZE without a launch."""
    from recurrent_state_quantization_gb300 import StatePool
    from recurrent_state_quantization_gb300 import _native as N
    dev = torch.device("cuda")
    P, Hh = 64, 128
    pool = StatePool(P, Hh, "int8", "scalar", 256, device=dev, k16=True)
    assert pool.split_scratch_bytes(P) > N.LS_SPLIT_STATIC_SCRATCH_BYTES
    slots = torch.arange(P, dtype=torch.int32, device=dev)
    x = torch.zeros(P, Hh, 128, device=dev)
    s = torch.zeros(P, Hh, device=dev)
    y = torch.full((P, Hh, 128), 7.0, device=dev)
    p = lambda t: C.c_void_p(t.data_ptr())
    rc = pool.lib.ls_decode_step_split_static(pool.handle, p(slots), P, p(x), p(x), p(x), p(s), p(s),
                                              p(y), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == N.LS_ERR_SIZE
    with pytest.raises(ValueError, match="static array holds"):
        pool.decode_step_split_static(slots, x, x, x, s, s, y=y)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())  # nothing ran
    # a batch that fits is accepted by the same pool
    small = pool.decode_step_split_static(slots[:8], x[:8], x[:8], x[:8], s[:8], s[:8])
    torch.cuda.synchronize()
    assert small.shape == (8, Hh, 128) and pool.status() == 0


def _c_call(pool, slots, x, y):
    """One ls_decode_step_split_static call through the C ABI, every buffer
    allocated beforehand by the caller."""
    p = lambda t: C.c_void_p(t.data_ptr())
    q, k, v, lam, beta = x
    return pool.lib.ls_decode_step_split_static(pool.handle, p(slots), int(slots.numel()), p(q), p(k),
                                                p(v), p(lam), p(beta), p(y),
                                                C.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_call_allocates_no_device_memory():
    """After one warm call (which loads the kernels), further calls leave the
    device's free memory unchanged: the scratch is the library's fixed array."""
    from recurrent_state_quantization_gb300 import _native as N
    a, b, slots, ins, _ = _twins("int8", "scalar", 3, 1)
    y = torch.empty(slots.numel(), b.H, 128, device=slots.device)
    assert _c_call(b, slots, ins[0], y) == N.LS_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    assert _c_call(b, slots, ins[1], y) == N.LS_OK  # closes the window: both kernels of the call
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert b.status() == 0


def test_static_scratch_refuses_another_current_device():
    """The array used is the one on the pool's device: with another device
    current the call returns LS_ERR_INVALID and launches nothing."""
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    from recurrent_state_quantization_gb300 import _native as N
    a, b, slots, ins, _ = _twins("deferred", "scalar", 5, 2)
    y = torch.full((slots.numel(), b.H, 128), 7.0, device=slots.device)
    with torch.cuda.device(1):
        assert _c_call(b, slots, ins[0], y) == N.LS_ERR_INVALID
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    assert _c_call(b, slots, ins[0], y) == N.LS_OK
