"""Host-side contracts that need no GPU: the product path fails loudly when
the CUDA library is missing (there is no fallback), and ``bench.py --impl
reference`` prints the reference arm's JSON line (the CPU oracle timed on
the host cores) with the keys the benchmark contract names."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from recurrent_state_quantization_gb300 import _native as N
    from recurrent_state_quantization_gb300 import pool
    monkeypatch.setattr(N, "LIB_PATH", str(tmp_path / "libls.so"))
    monkeypatch.setattr(N, "_lib", None)
    with pytest.raises(ImportError, match="libls.so is not built"):
        N.load()
    with pytest.raises(ImportError):
        pool.required_bytes(4, 2, "int8", "scalar", 16)
    with pytest.raises(ImportError):
        pool.StatePool(4, 2, "eager", device="cuda")


def _reference_line(env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_arm_json_line():
    lines = [ln for ln in _reference_line().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1 and d["higher_is_better"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"] and cb["nproc"] >= 1 and cb["host_cpu"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "gdn_serving_b256_h48_4pools"


def test_reference_arm_other_ranks_print_nothing():
    assert _reference_line({"RANK": "1", "WORLD_SIZE": "2"}).strip() == ""


def test_profiling_options_parse(monkeypatch):
    """The options the profiles' commands use: defaults leave the bench's own
    workload (W = 16 log variants, per-key-row INT8 without pairs)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.window is None and not a.col_scales and a.compensators == 0 and a.only is None
    monkeypatch.setattr(sys, "argv", ["bench.py", "--only", "int8", "--window", "8", "--col-scales",
                                      "--compensators", "4", "--pools", "1", "--ring", "2", "--no-extras"])
    a = bench.parse()
    assert (a.only, a.window, a.col_scales, a.compensators, a.pools, a.ring, a.no_extras) == \
        ("int8", 8, True, 4, 1, 2, True)
