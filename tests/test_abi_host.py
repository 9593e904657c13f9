"""Host-side checks of libls that need no GPU: the library loads, exports every
entry point include/ls.h declares, and validates descriptors and arguments
before touching CUDA."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from recurrent_state_quantization_gb300 import _native
    return _native.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ls.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ls_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for needed in ("ls_pool_create", "ls_decode_step", "ls_window_commit", "ls_pool_read"):
        assert needed in names


def test_every_declared_symbol_is_exported(lib):
    from recurrent_state_quantization_gb300 import _native
    names = declared_functions()
    assert sorted(_native.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def _desc(**kw):
    from recurrent_state_quantization_gb300 import _native as N
    d = dict(num_slots=4, num_heads=2, d_k=128, d_v=128, variant=N.LS_WINDOW_INT8,
             gate=N.LS_GATE_SCALAR, window=16, flags=0)
    d.update(kw)
    return N.LsDesc(**d)


def _bytes(lib, d):
    out = C.c_size_t(0)
    rc = lib.ls_pool_required_bytes(C.byref(d), C.byref(out))
    return rc, out.value


def test_required_bytes_layout(lib):
    from recurrent_state_quantization_gb300 import _native as N
    P, Hh, W = 4, 2, 16
    nh = P * Hh
    al = lambda x: (x + 255) // 256 * 256
    # eager: header + dense FP32 states
    rc, b = _bytes(lib, _desc(variant=N.LS_EAGER_FP32, window=0))
    assert rc == 0 and b == 256 + al(nh * 128 * 128 * 4)
    # INT8, scalar gate: INT8 base, scales, lbar, len, W entries (K, U, log-decay),
    # and the window-end queue of the tensor-core fold (16-byte header + one
    # (state index, request row) pair per state)
    rc, b = _bytes(lib, _desc())
    expect = (256 + al(nh * 128 * 128) + al(nh * 128 * 4) + al(nh * 4)
              + al(nh * 4) + 2 * al(nh * W * 128 * 4) + al(nh * ((W + 3) // 4 * 4) * 4)
              + al(16 + nh * 8))
    assert rc == 0 and b == expect
    # deferred, per-key gate
    rc, b = _bytes(lib, _desc(variant=N.LS_DEFERRED_FP32, gate=N.LS_GATE_PER_KEY))
    expect = (256 + al(nh * 128 * 128 * 4) + al(nh * 128 * 4) + al(nh * 4)
              + 3 * al(nh * W * 128 * 4))
    assert rc == 0 and b == expect


@pytest.mark.parametrize("field,value,code", [
    ("d_k", 64, -5), ("d_v", 256, -5), ("window", 0, -5), ("window", 257, -5),
    ("variant", 3, -1), ("gate", 2, -1), ("num_slots", 0, -1), ("num_heads", -1, -1),
    ("flags", 2, -1), ("flags", 0x80000000, -1)])
def test_bad_descriptors(lib, field, value, code):
    rc, _ = _bytes(lib, _desc(**{field: value}))
    assert rc == code


def test_column_scale_flag(lib):
    """LS_INT8_COLUMN_SCALES: INT8 pools only; one more [P*H][d_v] FP32 array
    (the value-column scales) after the key-row factors."""
    from recurrent_state_quantization_gb300 import _native as N
    P, Hh = 4, 2
    nh = P * Hh
    al = lambda x: (x + 255) // 256 * 256
    rc0, b0 = _bytes(lib, _desc())
    rc1, b1 = _bytes(lib, _desc(flags=N.LS_INT8_COLUMN_SCALES))
    # both formats keep the window-end queue of the tensor-core fold
    assert rc0 == 0 and rc1 == 0 and b1 == b0 + al(nh * 128 * 4)
    for variant in (N.LS_EAGER_FP32, N.LS_DEFERRED_FP32):
        rc, _ = _bytes(lib, _desc(variant=variant, flags=N.LS_INT8_COLUMN_SCALES))
        assert rc == N.LS_ERR_INVALID


def test_plain_update_flag(lib):
    """LS_PLAIN_UPDATE: the FP32 variants only; no extra memory."""
    from recurrent_state_quantization_gb300 import _native as N
    for variant in (N.LS_EAGER_FP32, N.LS_DEFERRED_FP32):
        rc0, b0 = _bytes(lib, _desc(variant=variant))
        rc1, b1 = _bytes(lib, _desc(variant=variant, flags=N.LS_PLAIN_UPDATE))
        assert rc0 == rc1 == 0 and b0 == b1
    rc, _ = _bytes(lib, _desc(flags=N.LS_PLAIN_UPDATE))
    assert rc == N.LS_ERR_INVALID


def test_bf16_key_flag(lib):
    """LS_LOG_BF16_K: log variants without compensator pairs; the key-side
    factors take 2 bytes instead of 4."""
    from recurrent_state_quantization_gb300 import _native as N
    P, Hh, W = 4, 2, 16
    nh = P * Hh
    al = lambda x: (x + 255) // 256 * 256
    for variant in (N.LS_DEFERRED_FP32, N.LS_WINDOW_INT8):
        rc0, b0 = _bytes(lib, _desc(variant=variant))
        rc1, b1 = _bytes(lib, _desc(variant=variant, flags=N.LS_LOG_BF16_K))
        assert rc0 == rc1 == 0
        assert b0 - b1 == al(nh * W * 128 * 4) - al(nh * W * 128 * 2)
    assert _bytes(lib, _desc(variant=N.LS_EAGER_FP32, flags=N.LS_LOG_BF16_K))[0] == N.LS_ERR_INVALID
    assert _bytes(lib, _desc(flags=N.LS_LOG_BF16_K | N.LS_INT8_COMPENSATORS(2)))[0] == N.LS_ERR_INVALID


def test_fp16_record_flag(lib):
    """LS_INT8_FP16_RECORDS: INT8 only, not with bfloat16 keys, compensator
    pairs allowed; keys and values of the log take 2 bytes each."""
    from recurrent_state_quantization_gb300 import _native as N
    P, Hh, W = 4, 2, 16
    nh = P * Hh
    al = lambda x: (x + 255) // 256 * 256
    for r in (0, 3):
        C = W + r
        rc0, b0 = _bytes(lib, _desc(flags=N.LS_INT8_COMPENSATORS(r)))
        rc1, b1 = _bytes(lib, _desc(flags=N.LS_INT8_COMPENSATORS(r) | N.LS_INT8_FP16_RECORDS))
        assert rc0 == rc1 == 0
        assert b0 - b1 == 2 * (al(nh * C * 128 * 4) - al(nh * C * 128 * 2))
    for variant in (N.LS_EAGER_FP32, N.LS_DEFERRED_FP32):
        assert _bytes(lib, _desc(variant=variant, flags=N.LS_INT8_FP16_RECORDS))[0] == N.LS_ERR_INVALID
    assert _bytes(lib, _desc(flags=N.LS_INT8_FP16_RECORDS | N.LS_LOG_BF16_K))[0] == N.LS_ERR_INVALID


def test_check_slots_flag(lib):
    """LS_CHECK_SLOTS: every variant and format; one int32 count per slot at
    the end of the layout, nothing else changes."""
    from recurrent_state_quantization_gb300 import _native as N
    P = 4
    al = lambda x: (x + 255) // 256 * 256
    for variant, flags in ((N.LS_EAGER_FP32, 0), (N.LS_DEFERRED_FP32, N.LS_LOG_BF16_K),
                           (N.LS_WINDOW_INT8, 0), (N.LS_WINDOW_INT8, N.LS_INT8_COLUMN_SCALES),
                           (N.LS_WINDOW_INT8, N.LS_INT8_COMPENSATORS(2) | N.LS_INT8_FP16_RECORDS)):
        rc0, b0 = _bytes(lib, _desc(variant=variant, flags=flags))
        rc1, b1 = _bytes(lib, _desc(variant=variant, flags=flags | N.LS_CHECK_SLOTS))
        assert rc0 == rc1 == 0 and b1 == b0 + al(P * 4)
    assert _bytes(lib, _desc(flags=N.LS_CHECK_SLOTS << 1))[0] == N.LS_ERR_INVALID


def test_compensator_flag(lib):
    """LS_INT8_COMPENSATORS(r): INT8 only, r <= 8; the log holds W + r entries
    (K, U, and the scalar-gate snapshots padded to 4)."""
    from recurrent_state_quantization_gb300 import _native as N
    P, Hh, W, r = 4, 2, 16, 4
    nh = P * Hh
    al = lambda x: (x + 255) // 256 * 256
    rc, b = _bytes(lib, _desc(flags=N.LS_INT8_COMPENSATORS(r)))
    C = W + r
    expect = (256 + al(nh * 128 * 128) + al(nh * 128 * 4) + al(nh * 4)
              + al(nh * 4) + 2 * al(nh * C * 128 * 4) + al(nh * ((C + 3) // 4 * 4) * 4))
    assert rc == 0 and b == expect
    rc, _ = _bytes(lib, _desc(flags=N.LS_INT8_COMPENSATORS(9)))
    assert rc == N.LS_ERR_INVALID
    rc, _ = _bytes(lib, _desc(variant=N.LS_DEFERRED_FP32, flags=N.LS_INT8_COMPENSATORS(1)))
    assert rc == N.LS_ERR_INVALID


def test_eager_ignores_window(lib):
    from recurrent_state_quantization_gb300 import _native as N
    rc, _ = _bytes(lib, _desc(variant=N.LS_EAGER_FP32, window=0))
    assert rc == 0


def test_null_arguments_are_rejected(lib):
    from recurrent_state_quantization_gb300 import _native as N
    assert lib.ls_pool_required_bytes(None, None) == N.LS_ERR_INVALID
    P = None
    assert lib.ls_decode_step(P, None, 1, None, None, None, None, None, None, None) == \
        N.LS_ERR_INVALID
    assert lib.ls_window_commit(P, None, 0, None) == N.LS_ERR_INVALID
    assert lib.ls_pool_read(P, None, 0, None, None) == N.LS_ERR_INVALID
    out = C.c_int32(0)
    assert lib.ls_pool_status(P, None, C.byref(out)) == N.LS_ERR_INVALID
    assert lib.ls_pool_destroy(None) == N.LS_OK
    d = _desc()
    h = C.c_void_p()
    assert lib.ls_pool_create(C.byref(d), None, 0, None, C.byref(h)) == N.LS_ERR_INVALID


def test_pool_create_checks_memory_before_cuda(lib):
    """Too few bytes or a misaligned pointer are refused on the host, before
    any CUDA call and without touching the memory (the pointer here is not a
    device pointer at all)."""
    from recurrent_state_quantization_gb300 import _native as N
    d = _desc()
    rc, need = _bytes(lib, d)
    assert rc == 0
    h = C.c_void_p()
    fake = C.c_void_p(1 << 20)
    assert lib.ls_pool_create(C.byref(d), fake, need - 1, None, C.byref(h)) == N.LS_ERR_SIZE
    assert lib.ls_pool_create(C.byref(d), C.c_void_p((1 << 20) + 16), need, None,
                              C.byref(h)) == N.LS_ERR_ALIGN
    assert not h.value


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -99):
        s = lib.ls_error_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    from recurrent_state_quantization_gb300 import _native as N
    assert lib.ls_abi_version() == N.LS_ABI_VERSION == 5


def test_split_entry_points_reject_null_before_any_launch(lib):
    from recurrent_state_quantization_gb300 import _native as N
    sz = C.c_size_t(7)
    assert lib.ls_split_scratch_bytes(None, 4, C.byref(sz)) == N.LS_ERR_INVALID
    assert sz.value == 7
    assert lib.ls_decode_step_split(None, None, 1, None, None, None, None, None, None, None, 0,
                                    None) == N.LS_ERR_INVALID
    assert lib.ls_decode_step_split_static(None, None, 1, None, None, None, None, None, None,
                                           None) == N.LS_ERR_INVALID


def test_product_path_does_not_import_the_oracle():
    """The package must not reach the CPU oracle (no fallback path)."""
    pkg = os.path.join(ROOT, "recurrent_state_quantization_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ls_oracle" not in text, f
