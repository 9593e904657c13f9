"""The byte model behind the roofline numbers, pinned to figures the pages print
(tests/golden/page_numbers.json, each with its source)."""
import json
import os

import pytest

from recurrent_state_quantization_gb300 import bytemodel as bm

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")))
MIB = 1024.0 ** 2


def g(key):
    return GOLD[key]["value"]


def test_dense_state_and_step_size():
    heads = 512 * 32
    assert heads * bm.state_bytes_fp32() / bm.GIB == pytest.approx(g("dense_state_gib_b512_h32"))
    assert heads * bm.eager_bytes("scalar") / bm.GIB == pytest.approx(
        g("dense_step_gib_b512_h32"), rel=0.02)


def test_dense_arith_intensity():
    # 4 d_k d_v FLOPs (decay + rank-1 update) over the dense read + write
    assert 4 * 128 * 128 / (2 * bm.state_bytes_fp32()) == g("dense_arith_intensity_fp32")


def test_dense_traffic_matches_profiled_gdn_b128():
    heads = 128 * 32
    read = heads * (bm.state_bytes_fp32() + bm.io_bytes("scalar") - 4 * 128) / bm.GIB
    write = heads * (bm.state_bytes_fp32() + 4 * 128) / bm.GIB
    assert read == pytest.approx(g("dense_dram_read_gib_gdn_b128"), rel=0.05)
    # the profiled write is a little below the state size (lines still dirty
    # in L2 when the kernel ends are not counted)
    assert write == pytest.approx(g("dense_dram_write_gib_gdn_b128"), rel=0.12)


def test_deferred_amortized_write_m8_16bit_keys():
    heads, M = 128 * 32, 8
    per_head = (bm.state_bytes_fp32() / M
                + (M - 1) / M * bm.entry_bytes("scalar", p_k=2, p_u=4) + 4 + 4 * 128)
    amort = heads * per_head / bm.GIB
    assert amort == pytest.approx(g("deltalog_amortized_write_gib_m8"), rel=0.25)
    dense_w = heads * (bm.state_bytes_fp32() + 4 * 128) / bm.GIB
    assert dense_w / amort == pytest.approx(g("deltalog_write_reduction_m8"), rel=0.15)


def test_leapquant_storage_figures():
    kib = bm.leapquant_record_buffer_bytes(16, "scalar") / 1024
    assert kib == pytest.approx(g("leapquant_fp16_buffer_kib_p16"), rel=0.01)
    bpe = bm.leapquant_boundary_bytes_per_elem()
    assert round(bpe, 2) == g("leapquant_bytes_per_elem")
    assert round(4 / bpe, 1) == g("leapquant_reduction_vs_fp32")


def test_stepquant_request_size():
    assert 48 * 48 * bm.state_bytes_fp32() / MIB == g("stepquant_mib_per_request")


def test_cycle_models_reduce_to_eager_at_m1():
    # M = 1: one base read and one base write per token, no log traffic
    assert bm.deferred_bytes("scalar", 1) == pytest.approx(bm.eager_bytes("scalar") + 8)
    assert bm.int8_bytes("scalar", 16) < bm.deferred_bytes("scalar", 16) < bm.eager_bytes("scalar")


def test_fp16_records_halve_the_record_bytes():
    """LeapQuant §4.3: a window of 16 FP16 records (k, u) of a 128 x 128 head
    takes about 8 KiB; a scalar-gate record is 2 d_k + 2 d_v bytes plus its
    FP32 decay snapshot, against 4 d_k + 4 d_v + 4 with FP32 records."""
    from recurrent_state_quantization_gb300 import bytemodel as bm
    assert bm.entry_bytes("scalar", p_k=2, p_u=2) == 516
    assert bm.entry_bytes("scalar") == 1028
    assert 16 * (bm.entry_bytes("scalar", p_k=2, p_u=2) - 4) == 8 * 1024
    W = 16
    full = bm.int8_bytes("scalar", W)
    half = bm.int8_bytes("scalar", W, p_k=2, p_u=2)
    assert full - half == ((W - 1) / W + (W - 1) / 2) * (1028 - 516)
