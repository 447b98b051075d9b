"""The reference arm of bench.py (the CPU oracle on a bounded sample) runs on
any machine and prints one JSON line with the keys the contract names, on
the same workload description as the GPU arm (CPU only)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    # the GPU arm's workload description, built from the same seeded workload
    import bench
    import workloads as W
    w = W.make_workload(bench.DEFAULT_CONFIG, W.config_seed(bench.DEFAULT_CONFIG), values=False)
    assert d["config"] == bench.decode_config(w, bench.DEFAULT_CONFIG, W.config_seed(bench.DEFAULT_CONFIG), 1)


def test_recorded_traffic_applies_only_to_the_captured_source(tmp_path):
    """roofline.traffic comes from a committed ncu summary only while the
    kernel's sources hash to the one it records; otherwise it is null."""
    import bench
    src = tmp_path / "kernel.cuh"
    src.write_text("// kernel v1\n")
    rec = tmp_path / "traffic.txt"
    rec.write_text(f"# note\nsource_sha: {bench.source_hash([str(src)])}\nbytes_per_launch[wl]: 12345\n")
    assert bench.recorded_traffic("wl", str(rec), [str(src)]) == 12345.0
    assert bench.recorded_traffic("other", str(rec), [str(src)]) is None
    src.write_text("// kernel v2\n")
    assert bench.recorded_traffic("wl", str(rec), [str(src)]) is None
    assert bench.recorded_traffic("wl", str(tmp_path / "missing.txt"), [str(src)]) is None

