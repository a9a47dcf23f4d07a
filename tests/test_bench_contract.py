"""bench.py's GPU arms keep the JSON contract: run on the CPU with stand-ins
for the CUDA pieces (tests/bench_fakes.py, the decoder computed by the
oracle), each arm must print one line with every required key.  The numbers
are meaningless here; the keys, units and launch counts are checked."""
import json
import os
import subprocess
import sys

import pytest

pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKES = os.path.join(ROOT, "tests", "bench_fakes.py")

TOP = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
       "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"}


def run_arm(*args):
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, FAKES, *args], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def check_common(line, steps, warmup):
    assert TOP <= set(line), TOP - set(line)
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["n_gpus"] == 1 and line["steps"] == steps and line["warmup"] == warmup
    assert line["vs_baseline"] is None and line["dtype"] == "f32"
    assert line["config"]["workload"] == "tiny"
    roof = line["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(roof)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["unit"] == "tokens/s" and cpu["sample"]
    e2e = line["e2e"]
    assert set(e2e) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"} and e2e["unit"] == "tokens/s"
    assert set(line["clocks"]) == {"sm_mhz", "sm_max_mhz", "reasons"}


def test_decode_batch_one_line():
    line = run_arm("--workload", "tiny", "--steps", "12", "--warmup", "3", "--cpu-budget", "0.5")
    check_common(line, 12, 3)
    assert line["metric"].startswith("decode tokens/s at batch 1")
    assert line["roofline"]["bound"] == "hbm" and line["roofline"]["unit"] == "GB/s"
    assert "GEMV_W13" in line["roofline"]["kernel"]
    assert line["gpu_launches"] == 12 * (5 * 5 + 1)  # tiny: 5 layers
    assert line["e2e"]["d2h_bytes_per_step"] == 4 * 512 and line["e2e"]["h2d_bytes_per_step"] == 1232
    assert set(line["per_position"]) == {"2", "129", "505"}


def test_decode_batch_sixteen_line():
    line = run_arm("--workload", "tiny", "--batch", "16", "--steps", "4", "--warmup", "3", "--cpu-budget", "0.5")
    check_common(line, 4, 3)
    assert "at batch 16" in line["metric"] and line["config"]["batch"] == 16
    assert line["gpu_launches"] == 4 * (5 * 5 + 2)  # the embedding kernel on the tensor-core path
    assert line["e2e"]["d2h_bytes_per_step"] == 16 * 4 * 512


def test_prefill_line():
    line = run_arm("--workload", "tiny", "--prefill", "130", "--steps", "2", "--warmup", "3", "--cpu-budget", "0.5")
    check_common(line, 2, 3)
    assert line["metric"].startswith("prefill tokens/s of a 130-token prompt")
    assert line["config"]["prefill_tokens"] == 130
    assert line["gpu_launches"] == 2 * (2 * (5 * 5 + 2) + (5 * 5 + 1))  # chunks of 64, 64 and 2 rows
    assert line["e2e"]["h2d_bytes_per_step"] == 3 * 1232


def test_decode_line_per_config_block():
    line = run_arm("--workload", "tiny", "--steps", "4", "--warmup", "3", "--cpu-budget", "0.5", "--no-positions",
                   "--per-config", "tiny,tiny:4", "--per-config-runs", "2")
    check_common(line, 4, 3)
    pc = line["per_config"]
    assert set(pc) == {"tiny", "tiny_b4", "_peak"}
    for key, B, steps in (("tiny", 1, 128), ("tiny_b4", 4, 128)):
        e = pc[key]
        assert e["batch"] == B and e["steps"] == steps
        assert e["tokens_per_s"] == pytest.approx(B * steps / (e["ms_per_step"] * steps / 1000.0))
        assert e["frac_of_measured"] == pytest.approx(e["gbs"] / line["roofline"]["peak"])
        assert e["l2_resident"] is True and e["launches_per_step"] == 5 * 5 + 1
    # the default run of a small workload reports no per-config block
    assert run_arm("--workload", "tiny", "--steps", "2", "--warmup", "3", "--cpu-budget", "0.2",
                   "--no-positions")["per_config"] is None
