"""bench.py's reference arm on the host cores: it times the fp64 oracle on the
workload it is given and prints one JSON line with the keys the benchmark line
carries (no GPU involved)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "single_head_n128_d64_causal", "--steps", "3", "--warmup", "3"],
        cwd=ROOT, capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["config"]["workload"] == "single_head_n128_d64_causal"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def test_peak_follows_the_sampled_clock():
    b = _bench()
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sustained_sm_mhz": 1450.0,
             "sm_max_mhz": 2070.0, "hbm_gbs": 6800.0, "source": "measured"}
    at_max = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0}
    assert b.tensor_peak(peaks, at_max)[0] == 1900.0                      # burst at max clock
    assert b.tensor_peak(peaks, {"sm_mhz": 2025.0, "sm_max_mhz": 2070.0})[0] == 1900.0
    assert b.tensor_peak(peaks, {"sm_mhz": 1460.0, "sm_max_mhz": 2070.0})[0] == 1700.0
    mid = b.tensor_peak(peaks, {"sm_mhz": 1950.0, "sm_max_mhz": 2070.0})[0]
    assert abs(mid - 1900.0 * 1950.0 / 2070.0) < 1e-9                      # scaled in between
    assert b.tensor_peak(peaks, {"sm_mhz": None, "sm_max_mhz": None})[0] == 1900.0


def test_visible_pairs_counts_the_causal_triangle():
    b = _bench()
    brute = lambda n, m, c: sum(1 for q in range(n) for k in range(m) if not c or k <= q)
    for n, m in ((1, 1), (5, 5), (7, 3), (3, 7), (128, 128)):
        for causal in (False, True):
            assert b.visible_pairs(n, m, causal) == brute(n, m, causal), (n, m, causal)
    assert b.visible_pairs(4096, 4096, True) * 64 == 537_001_984  # 5.37e8 at the benchmark shape


def test_io_model_counts_the_score_matrices():
    b = _bench()
    m = b.io_model_bytes(1, 2, 1024, 1024, 128)
    io = 2 * ((2 * 1024 + 2 * 1024) * 128 * 2 + 1024 * 4)      # Q, K, V, O bf16; L fp32
    assert m["tiled"] == io
    assert m["standard"] - m["tiled"] == 2 * 4 * 1024 * 1024 * 2  # write S, read S, write P, read P
    rows = b.io_configs()
    assert {r[3] for r in rows} == {1024, 4096, 16384}
    assert all(r[1] * r[2] * r[3] in (r[3], b.IO_QUERY_ROWS) for r in rows)
