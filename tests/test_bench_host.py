"""Host side of the benchmark, without a GPU.

The multi-rank path runs one independent replica per rank: the only exchange
is the slowest rank's time, taken with an all-reduce MAX after the timed
region.  Checked here with two ``gloo`` ranks on the CPU.  The reference arm
(the oracle on the host cores) runs on rank 0 alone and prints one JSON line
carrying the same metric and config keys as the GPU arm; other ranks exit 0
without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world, device="cpu")
        rate = bench.job_rate(100, world, slowest)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo(tmp_path):
    times = [0.25, 0.75]
    mp.start_processes(_rank_main, args=(2, _free_port(), times, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        got = json.loads((tmp_path / f"r{r}.json").read_text())
        assert got["slowest"] == 0.75  # every rank sees the slowest rank's time
        assert got["rate"] == pytest.approx(2 * 100 / 0.75)  # all ranks' units over it


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_rate(64, 1, 2.0) == 32.0


def _run(args, **env):
    e = dict(os.environ, OMP_NUM_THREADS="2", **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=e, capture_output=True,
                          text=True, timeout=300)


@pytest.mark.parametrize("batch", [1, 3])
def test_reference_arm_line(batch):
    r = _run(["--impl", "reference", "--workload", "tiny", "--batch", str(batch), "--steps", "6", "--warmup", "3",
              "--reference-budget", "5"])
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.metric_of(batch)
    assert line["config"]["workload"] == "tiny" and line["config"]["batch"] == batch
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["steps"] == 6 and line["warmup"] == 3 and line["value"] > 0
    assert line["ms_per_step"] == pytest.approx(1000.0 * batch / line["value"], rel=1e-9)
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == line["value"] and cpu["cores"] == 2
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_prefill_line():
    r = _run(["--impl", "reference", "--workload", "tiny", "--prefill", "100", "--reference-budget", "5"])
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["metric"] == bench.metric_of(1, prefill=100)
    assert line["config"]["prefill_tokens"] == 100 and line["config"]["chunk_rows"] == bench.PREFILL_CHUNK
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_prefill_chunks_and_bytes():
    assert bench.prefill_chunks(130) == [(0, 64), (64, 64), (128, 2)]
    assert bench.prefill_chunks(64) == [(0, 64)]
    wl = bench.WORKLOADS["tiny"]
    # each chunk: the weights once, and the cache rows up to its last position once
    want = 3 * bench.weight_bytes(wl) + sum(bench.kv_bytes(wl, p) for p in (63, 127, 129))
    assert bench.prefill_bytes(wl, 130) == want


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--workload", "tiny"], RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.parametrize("args", [["--warmup", "2"], ["--batch", "65"], ["--weights", "bf16", "--batch", "4"],
                                  ["--workload", "tiny", "--layers", "6"], ["--workload", "tiny", "--prefill", "513"],
                                  ["--workload", "tiny", "--prefill", "64", "--batch", "2"]])
def test_bench_rejects_invalid_runs(args):
    r = _run(["--impl", "reference", *args])
    assert r.returncode == 2 and "error" in r.stderr


def test_metric_names_the_batch():
    assert bench.metric_of(1) == bench.METRIC
    assert "at batch 16" in bench.metric_of(16)
    assert "bf16 weights" in bench.metric_of(1, bf16=True)
