"""The allocation-free split-replay step (ls_decode_step_split_static, its
coefficient scratch in the library's fixed device array) against the
caller-scratch entry point (ls_decode_step_split): twin pools, two calls in a
row, the same bits in y and in the pools.  Collected last so that it also
runs after every other GPU test in the same process."""
import ctypes as C

import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


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
