"""bench.py's reference arm on the CPU: the one JSON line and the keys the
measurement contract asks for, on the tiny workload so it runs in seconds."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "0"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["warmup"] >= 3 and d["steps"] == 2 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert isinstance(cb["sample"], str) and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the time per step is the workload's tokens at the reported rate
    assert abs(d["ms_per_step"] - 1000.0 * d["config"]["T"] / d["value"]) < 1e-6 * d["ms_per_step"]
    assert d["ms_per_step_kind"].startswith("extrapolated")
    assert cb["extrapolated_step_s"] > 0 and 0 < cb["sample_s"]


def test_span_summary_arithmetic():
    """The e2e diagnostic's overlap bookkeeping on hand-made spans: passes of
    10 ms back to back with 2 ms gaps, copies of 6 ms starting 1 ms after
    each pass ends."""
    sys.path.insert(0, ROOT)
    import bench

    fwd = [(0.0, 10.0), (12.0, 22.0), (24.0, 34.0)]
    cpy = [(11.0, 17.0), (23.0, 29.0), (35.0, 41.0)]
    s = bench.span_summary(fwd, cpy)
    assert s["prompts"] == 3 and s["span_ms"] == 41.0
    assert s["forward_ms_mean"] == 10.0 and s["copy_ms_max"] == 6.0
    assert s["compute_idle_ms_total"] == 4.0
    assert s["copy_start_after_ready_ms_mean"] == 1.0
    assert s["copy_overlapped_with_next_forward_ms_total"] == 10.0   # 5 + 5


def test_expected_miss_follows_the_oracle_mode():
    """The stated-bar tests mark a bar as an expected failure exactly where the
    oracle's own rounding mode (the library's rounding points) misses it; the
    float32 path never gets one."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity_record import expected_miss, load_golden

    golden = {"workloads": {"w": {"modes": {
        "bf16_fused": {"free_max": 9e-3, "forced_max": 1e-3, "logit_max_abs": 0.06,
                       "argmax_agreement": 0.996},
        "tf32": {"free_max": 1e-3, "forced_max": 5e-4, "logit_max_abs": 0.01,
                 "argmax_agreement": 0.99}}}}}
    assert "free_max" in expected_miss(golden, "w", "bf16", "layer_free")
    assert expected_miss(golden, "w", "bf16", "layer_forced") is None
    assert "0.06" in expected_miss(golden, "w", "bf16", "logit_max_abs")
    assert expected_miss(golden, "w", "bf16", "argmax_raw") is None
    assert expected_miss(golden, "w", "tf32", "argmax_raw") is not None
    assert expected_miss(golden, "w", "tf32", "layer_free") is None
    assert all(expected_miss(golden, "w", "f32", b) is None
               for b in ("layer_free", "layer_forced", "logit_max_abs", "argmax_raw"))
    assert expected_miss(golden, "other", "bf16", "layer_free") is None
    # the committed file covers every model workload in both rounding modes
    real = load_golden()
    for name in ("tiny", "small", "qwen3-0.6b-shape", "qwen3-8b-shape"):
        assert {"bf16", "bf16_fused", "tf32"} <= set(real["workloads"][name]["modes"])
