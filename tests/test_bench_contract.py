"""The benchmark's reference arm on the CPU (no GPU needed): one JSON line with
the keys the harness reads, the oracle timed on a bounded sample.  The 12-layer
decode workload keeps this quick (the mixed step's sample takes about 90 s to
prepare); the code path is the same for every workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "decode12", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 1
    assert "workload" in d["config"]
    # the same config keys as the GPU arm prints for this workload (the driver compares them)
    for key in ("pool_slots", "layers", "heads", "head_size", "decode_slots", "state_dtype",
                "input_dtype", "output_dtype", "parallelism", "l2", "graph"):
        assert key in d["config"], key
    assert d["config"]["parallelism"] == "1 gpu" and d["config"]["graph"] is False
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_has_no_host_copy_reference_for_hibernate():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "hibernate", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads([ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")][-1])
    assert d["impl"] == "reference" and "unavailable" in d


def test_output_dtype_reaches_both_arms_configs():
    """--out-dtype names the mixed step's output dtype in the config both arms print
    (the GPU arm's Mixed.config and the reference arm's shapes-only copy share it)."""
    sys.path.insert(0, ROOT)
    import bench
    for od in ("f32", "bf16"):
        args = bench.parse_args(["--impl", "reference", "--out-dtype", od])
        cfg = bench._shapes_only(args).config()
        assert cfg["output_dtype"] == od
        assert cfg["workload"].endswith("; bf16 outputs") == (od == "bf16")
    args = bench.parse_args(["--impl", "reference", "--workload", "decode12", "--out-dtype", "bf16"])
    assert bench._shapes_only(args).config()["output_dtype"] == "f32"  # mixed step only
