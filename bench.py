#!/usr/bin/env python3
"""Decode benchmark: tokens/s and HBM-roofline fraction of the batch-1 decode
step on one GB300 (default workload: the Llama-2-7B shape in fp32).

A step is one forward(token, pos) -> logits over the whole model.  Warm-up
steps decode positions 0..W-1, the timed steps positions W..W+K-1 of one
teacher-forced stream of seeded uniform tokens (positions wrap to 0, with the
cache rewound, after seq_len).  The weights (26.4 GB at the 7B shape) are far
larger than L2, so every step streams them from HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores on the same workload instead (a bounded sample of steps).
Multi-GPU (torchrun): each rank runs an independent replica, no collective on
the data path; value = all ranks' tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import WORKLOADS  # noqa: E402

METRIC = "decode tokens/s at batch 1 and % of HBM roofline (GB/s vs ~8 TB/s), 1 GB300"
TC_MIN_BATCH = 16  # steps of this many rows run their matrix products on the tensor cores
NOMINAL_HBM_GBS = 8000.0
READ_CEILING_GBS = 7250.0  # pure bulk-copy read stream on GB300 (see the roofline's read_ceiling)
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the dominant kernel (rmsnorm + W1/W3 + SwiGLU at the 7B shape), per weight
# type, from one ncu capture of that kernel: (bytes per launch, the sha256
# prefixes of gemv.cu it holds for).  The fp32 figure was taken on source
# 4177b02e...; 5474aa3e... changed only the bf16 branches of the kernel template
# (`if (WT)`, compiled out of the fp32 kernel), so the fp32 kernel is the same.
W13_NCU_TRAFFIC = {
    "f32": (363956480, ("4177b02e97bce001", "5474aa3edc02e859")),
    "bf16": (183838976, ("5474aa3edc02e859",)),
}


def weight_bytes(wl, wb: int = 4) -> int:
    """Weight bytes one step streams: every matrix (wb bytes per weight: 4
    fp32, 2 bf16), the RMSNorm gains, the classifier, one embedding row (fp32)."""
    d, h, L, kv, V = wl.dim, wl.hidden_dim, wl.n_layers, wl.kv_dim, wl.vocab_size
    return wb * (L * (2 * d * d + 2 * kv * d + 3 * d * h) + V * d) + 4 * (L * 2 * d + 2 * d)


def kv_bytes(wl, pos: int) -> int:
    """K and V cache bytes one step at ``pos`` reads."""
    return 4 * wl.n_layers * 2 * wl.kv_dim * (pos + 1)


def w13_bytes(wl, wb: int = 4) -> int:
    """Algorithmic bytes of one rmsnorm+W1/W3+SwiGLU launch: both matrices
    (wb bytes per weight), the gain vector, x in and hb out."""
    return wb * 2 * wl.hidden_dim * wl.dim + 4 * (2 * wl.dim + wl.hidden_dim)


PREFILL_CHUNK = 64  # rows of one prefill step (l2_prefill's chunk without L2_FLAG_DEBUG)


def prefill_chunks(T: int) -> list:
    """(first position, rows) of each chunk of a T-token prompt from position 0."""
    return [(c0, min(PREFILL_CHUNK, T - c0)) for c0 in range(0, T, PREFILL_CHUNK)]


def prefill_bytes(wl, T: int) -> int:
    """Algorithmic bytes of a T-token prefill: each chunk streams the weights
    once and reads the cache rows up to its last position once."""
    return sum(weight_bytes(wl) + kv_bytes(wl, c0 + r - 1) for c0, r in prefill_chunks(T))


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except OSError:
        return {}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def config_of(wl, batch: int = 1, bf16: bool = False) -> dict:
    return {"workload": wl.name, "dim": wl.dim, "hidden_dim": wl.hidden_dim, "n_layers": wl.n_layers,
            "n_heads": wl.n_heads, "n_kv_heads": wl.n_kv_heads, "vocab_size": wl.vocab_size,
            "seq_len": wl.seq_len, "batch": batch, "parallelism": "replicas",
            "weights": "seeded random (synth)", "tokens": "seeded uniform, teacher-forced",
            "l2": "inputs larger than L2" if weight_bytes(wl) > 129e6 else "weights fit in L2 (effective bandwidth)",
            "gemv": gemv_path(batch, bf16)}


def on_tensor_cores(batch: int, bf16: bool = False) -> bool:
    """Steps of this many rows run their matrix products on the tensor cores (all
    steps of several rows with bf16 weights)."""
    return batch >= TC_MIN_BATCH or (bf16 and batch > 1)


def gemv_path(batch: int, bf16: bool = False) -> str:
    if on_tensor_cores(batch, bf16):
        return ("tensor cores (tcgen05 kind::f16: bf16 weights, inputs in three bf16 parts: exact products)" if bf16 else
                "tensor cores (tcgen05 kind::tf32, 3-term hi/lo split: fp32-level products)")
    return "CUDA cores (bf16 weights widened to fp32, fp32 FMA)" if bf16 else "CUDA cores (fp32 FMA)"


def load_weights_device(wl, keep_host: bool):
    """Device tensors of the workload's weights; host arrays too if asked."""
    import torch
    if keep_host:
        host = synth.make_weights(wl)
        import llama_transformer_decode_gb300 as pkg
        return pkg.to_device(host), host
    dev = {}
    chunk = 1 << 26
    buf = torch.empty(chunk, dtype=torch.float32, pin_memory=True)
    bnp = buf.numpy()
    for name in wl.tensor_names():
        if name == "wcls" and wl.shared_wcls:
            dev["wcls"] = dev["emb"]
            continue
        t = torch.empty(wl.shape(name), dtype=torch.float32, device="cuda")
        flat = t.view(-1)
        for st in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - st)
            synth.fill_range(wl, name, st, bnp[:n])
            flat[st:st + n].copy_(buf[:n], non_blocking=False)
        dev[name] = t
    return dev, None


def host_threads() -> int:
    """Threads the oracle's parallel loops run on."""
    import oracle
    return oracle.num_threads()


def metric_of(batch: int, bf16: bool = False, prefill: int = 0) -> str:
    if prefill:
        return (f"prefill tokens/s of a {prefill}-token prompt and % of HBM roofline "
                "(GB/s vs ~8 TB/s), 1 GB300")
    tail = " with bf16 weights" if bf16 else ""
    return METRIC.replace("at batch 1", f"at batch {batch}{tail}")


def max_over_ranks(v: float, world: int, device: str = "cuda") -> float:
    """The largest of the ranks' values (each rank passes its own)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, slowest_s: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / slowest_s


def oracle_rate(wl, host_w, tokens, budget_s: float, min_steps: int = 2):
    """Teacher-forced oracle steps from position 0 until the time budget is
    spent; returns (steps, seconds, threads)."""
    import oracle
    m = oracle.Model(wl.config_tuple(), host_w)
    t0 = time.perf_counter()
    n = 0
    while n < len(tokens) and (n < min_steps or time.perf_counter() - t0 < budget_s):
        m.forward(int(tokens[n]), n)
        n += 1
    el = time.perf_counter() - t0
    return n, el, host_threads()


def run_reference(args, wl):
    """The oracle on the host cores, on the same workload, batch and staggered
    positions as the GPU arm: each step is one forward per slot."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0  # one CPU baseline per job, taken on rank 0
    if args.prefill:
        return run_reference_prefill(args, wl, world)
    import oracle
    B, S = args.batch, wl.seq_len
    host_w = synth.make_weights(wl)
    m = oracle.Model(wl.config_tuple(), host_w, n_slots=B)
    streams = [synth.token_stream(wl, b, S) for b in range(B)]
    offsets = [b * S // B for b in range(B)]
    for b in range(B):
        if offsets[b]:
            m.key_cache[b][:, : offsets[b]] = synth.kv_rows(wl, b, offsets[b], "k")
            m.value_cache[b][:, : offsets[b]] = synth.kv_rows(wl, b, offsets[b], "v")

    def step(s):
        for b in range(B):
            p = (offsets[b] + s) % S
            if p == 0 and s > 0:  # the slot wraps: its cache starts over
                m.key_cache[b][:] = 0
                m.value_cache[b][:] = 0
            m.forward(int(streams[b][p]), p, slot=b)

    for s in range(args.warmup):
        step(s)
    # size the timed sample from one step's cost so the run stays within the budget
    t0 = time.perf_counter()
    step(args.warmup)
    one = time.perf_counter() - t0
    k = max(1, min(args.steps, int(args.reference_budget / max(one, 1e-6))))
    first = args.warmup + 1
    t0 = time.perf_counter()
    for s in range(first, first + k):
        step(s)
    el = time.perf_counter() - t0
    value = B * k / el
    where = (f"positions {first % S}..{(first + k - 1) % S}" if B == 1 else
             f"slot b from floor(b*{S}/{B}) + {first}, wrapping at {S}")
    sample = (f"{k} teacher-forced oracle steps of {wl.name} ({B} sequence{'s' if B > 1 else ''}) at {where} "
              f"(of {args.steps} requested), after {first} untimed")
    cfg = config_of(wl, B)
    cfg["gemv"] = "oracle: fp32 storage, double accumulation, OpenMP rows"
    line = {"impl": "reference", "metric": metric_of(B), "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": k, "warmup": args.warmup, "ms_per_step": 1000.0 * el / k, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate/f32-storage", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": host_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference_prefill(args, wl, world: int):
    """The oracle on the same prompt, one teacher-forced step per token from
    position 0, for as many tokens as the time budget allows."""
    import oracle
    T = args.prefill
    host_w = synth.make_weights(wl)
    toks = synth.token_stream(wl, 0, T)
    m = oracle.Model(wl.config_tuple(), host_w)
    for p in range(min(args.warmup, T)):  # untimed
        m.forward(int(toks[p]), p)
    n, el, threads = oracle_rate(wl, host_w, toks, args.reference_budget)
    value = n / el
    cfg = config_of(wl, 1)
    cfg.update({"prefill_tokens": T, "chunk_rows": PREFILL_CHUNK, "positions": f"0..{T - 1}",
                "gemv": "oracle: fp32 storage, double accumulation, OpenMP rows"})
    sample = f"the first {n} of the prompt's {T} tokens, one oracle step each, after {min(args.warmup, T)} untimed"
    line = {"impl": "reference", "metric": metric_of(1, prefill=T), "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": 1, "warmup": args.warmup, "ms_per_step": 1000.0 * el,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate/f32-storage",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# Every workload's own throughput, reported beside the headline line: the
# small decoders over their full teacher-forced runs, and the batched workload
# at one, 16 and 64 sequences.
DEFAULT_PER_CONFIG = "tiny,gqa_small,mid,batched_1b,batched_1b:16,batched_1b:64"
BATCHED_PER_CONFIG_STEPS = 256
L2_BYTES = 129e6  # the GPU's L2 cache: weights below this stay resident between steps


def parse_per_config(spec: str) -> list:
    """[(workload, batch)] from "name[:B],..." ("none": no entries)."""
    if not spec or spec == "none":
        return []
    out = []
    for item in spec.split(","):
        name, _, b = item.strip().partition(":")
        if name not in WORKLOADS:
            raise ValueError(f"unknown workload {name!r} in --per-config")
        B = int(b) if b else 1
        if not 1 <= B <= 64:
            raise ValueError(f"batch {B} outside 1..64 in --per-config")
        out.append((name, B))
    return out


def per_config_rates(entries, hbm: float, peak_src: str, runs: int) -> dict:
    """Tokens/s and HBM bandwidth of each (workload, batch), each on its own
    decoder and stream, timed with CUDA events after an untimed pass that
    builds its graphs.  Batch 1: the workload's full teacher-forced run from
    position 0, `runs` times (the cache rewound each run), median reported.
    Batches: slot b starts at floor(b * seq_len / B) (earlier rows imported) and
    steps BATCHED_PER_CONFIG_STEPS times, wrapping at the end of the context;
    `runs` consecutive segments, median reported."""
    import torch

    import llama_transformer_decode_gb300 as pkg
    out = {}
    loaded = {}
    for name, B in entries:
        wl = WORKLOADS[name]
        if name not in loaded:
            loaded.clear()
            loaded[name] = load_weights_device(wl, keep_host=False)[0]
        w = loaded[name]
        stream = torch.cuda.Stream()
        dec = pkg.Decoder(wl.config_tuple(), w, max_batch=B, stream=stream)
        S = wl.seq_len
        batched = B > 1 or name == "batched_1b"
        n = min(BATCHED_PER_CONFIG_STEPS, S) if batched else min(wl.steps or S, S)
        offsets = [b * S // B for b in range(B)]
        streams = [synth.token_stream(wl, b, S) for b in range(B)]
        logits = torch.empty((B, wl.vocab_size), device="cuda")

        def prepare():
            dec.reset()
            for b in range(B):
                if offsets[b]:
                    dec.kv_import(synth.kv_rows(wl, b, offsets[b], "k"), synth.kv_rows(wl, b, offsets[b], "v"),
                                  slot=b)

        def steps(first, count):
            for st in range(first, first + count):
                pos = [(offsets[b] + st) % S for b in range(B)]
                for b in range(B):
                    if pos[b] == 0 and dec.position(b) > 0:
                        dec.reset(b)
                if B == 1:
                    dec.forward(int(streams[0][pos[0]]), pos[0], logits[0])
                else:
                    dec.forward_batch([int(streams[b][pos[b]]) for b in range(B)], pos, logits)
            return [[(offsets[b] + st) % S for b in range(B)] for st in range(first, first + count)]

        prepare()
        steps(0, min(n, 8))  # untimed: builds the graphs
        dec.sync()
        times, byts = [], []
        if not batched:
            for _ in range(runs):
                prepare()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                pos = steps(0, n)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1) / 1000.0)
                byts.append(sum(weight_bytes(wl) + sum(kv_bytes(wl, p) for p in ps) for ps in pos))
            where = f"0..{n - 1}, {runs} runs"
        else:
            prepare()
            seg = max(1, n // runs)
            for r in range(runs):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                pos = steps(r * seg, seg)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1) / 1000.0)
                byts.append(sum(weight_bytes(wl) + sum(kv_bytes(wl, p) for p in ps) for ps in pos))
            n = seg
            where = (f"slot b from floor(b*{S}/{B}), {runs} segments of {seg} steps" if B > 1 else
                     f"0..{runs * seg - 1} in {runs} segments of {seg} steps")
        dec.sync()
        order = sorted(range(len(times)), key=lambda i: times[i])
        mid = order[len(order) // 2]
        t, by = times[mid], byts[mid]
        gbs = by / t / 1e9
        key = name if B == 1 and name != "batched_1b" else f"{name}_b{B}"
        out[key] = {
            "batch": B, "tokens_per_s": B * n / t, "ms_per_step": 1000.0 * t / n, "steps": n, "positions": where,
            "gbs": gbs, "frac_of_measured": gbs / hbm, "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
            "bytes_per_step_avg": by / n, "l2_resident": weight_bytes(wl) < L2_BYTES,
            "launches_per_step": dec.kernels_per_step(B),
            "gemv": gemv_path(B)}
        dec.close()
    loaded.clear()
    out["_peak"] = f"{hbm:.1f} GB/s {peak_src} (MEASURED_PEAKS.json hbm_gbs); timing: CUDA events, median of {runs}"
    return out


def fp32_alu_peak_tflops(props) -> float:
    """fp32 FMA peak: SMs x 128 lanes x 2 flop x the maximum SM clock."""
    peaks = measured_peaks()
    mhz = peaks.get("sm_max_mhz", 2070.0)
    return props.multi_processor_count * 128 * 2 * mhz * 1e6 / 1e12


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import llama_transformer_decode_gb300 as pkg

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    pkg._native.load()
    props = torch.cuda.get_device_properties(local_rank)
    uuid = str(props.uuid)
    B = args.batch
    bf16 = args.weights == "bf16"
    wb = 2 if bf16 else 4

    cpu_leg = rank == 0 and world == 1 and not args.no_cpu
    w_dev, host_w = load_weights_device(wl, keep_host=cpu_leg)
    stream = torch.cuda.Stream()
    dec = pkg.Decoder(wl.config_tuple(), w_dev, max_batch=B, stream=stream,
                      flags=pkg.L2_FLAG_BF16_WEIGHTS if bf16 else 0)
    S = wl.seq_len
    streams = [synth.token_stream(wl, b, S) for b in range(B)]
    out = torch.empty((B, wl.vocab_size), device="cuda")
    kern = dec.kernels_per_step(B)
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs")
    peak_src = "of measured" if hbm else "of fallback"
    hbm = hbm or FALLBACK_HBM_GBS

    # Slot b starts at floor(b * S / B) (0 for a batch of one) and wraps to 0,
    # with its cache rewound, at the end of the context.
    offsets = [b * S // B for b in range(B)]
    for b in range(B):
        if offsets[b]:
            # rows before the offset stand for tokens decoded earlier; their
            # values do not change a step's cost, so they are imported
            dec.kv_import(synth.kv_rows(wl, b, offsets[b], "k"), synth.kv_rows(wl, b, offsets[b], "v"), slot=b)

    def positions(step):
        return [(offsets[b] + step) % S for b in range(B)]

    def run_steps(first, n, host_out=None):
        for s in range(first, first + n):
            pos = positions(s)
            for b in range(B):
                if pos[b] == 0 and dec.position(b) > 0:
                    dec.reset(b)
            if B == 1:
                if host_out is None:
                    dec.forward(int(streams[0][pos[0]]), pos[0], out[0])
                else:
                    dec.forward_host(int(streams[0][pos[0]]), pos[0], host_out)
            else:
                dec.forward_batch([int(streams[b][pos[b]]) for b in range(B)], pos, out)
                if host_out is not None:
                    stream.synchronize()
                    host_out[...] = out.cpu().numpy()

    def barrier():
        if world > 1:
            dist.barrier()

    run_steps(0, args.warmup)
    dec.sync()

    # ---- device-resident timed region ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(uuid) as clocks:
        ev0.record(stream)
        run_steps(args.warmup, args.steps)
        ev1.record(stream)
        ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    dec.sync()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    value = job_rate(B * args.steps, world, ms / 1000.0)
    timed_pos = [positions(s) for s in range(args.warmup, args.warmup + args.steps)]
    bytes_total = sum(weight_bytes(wl, wb) + sum(kv_bytes(wl, p) for p in pos) for pos in timed_pos)
    step_gbs = bytes_total / (ms / 1000.0) / 1e9

    # ---- rate at chosen positions (cache rows before them imported) ----
    per_pos = {}
    if B == 1 and not args.no_positions:
        for p0 in (0, S // 4 - 1, S - 9):
            dec.reset()
            if p0:
                dec.kv_import(synth.kv_rows(wl, 0, p0, "k"), synth.kv_rows(wl, 0, p0, "v"))
            for p in range(p0, p0 + 2):
                dec.forward(int(streams[0][p]), p, out[0])
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for p in range(p0 + 2, p0 + 8):
                dec.forward(int(streams[0][p]), p, out[0])
            a1.record(stream)
            a1.synchronize()
            t = a0.elapsed_time(a1) / 6
            gb = sum(weight_bytes(wl, wb) + kv_bytes(wl, p) for p in range(p0 + 2, p0 + 8)) / 6
            per_pos[str(p0 + 2)] = {"tokens_per_s": 1000.0 / t, "ms_per_step": t, "gbs": gb / t / 1e6}
        dec.sync()

    # ---- end to end through the public call with host output ----
    host_logits = np.empty(wl.vocab_size if B == 1 else (B, wl.vocab_size), np.float32)
    dec.reset()
    for b in range(B):
        if offsets[b]:
            dec.kv_import(synth.kv_rows(wl, b, offsets[b], "k"), synth.kv_rows(wl, b, offsets[b], "v"), slot=b)
    run_steps(0, args.warmup, host_logits)
    barrier()
    t0 = time.perf_counter()
    run_steps(args.warmup, args.steps, host_logits)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": job_rate(B * args.steps, world, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": dec.step_input_bytes(),
           "d2h_bytes_per_step": 4 * wl.vocab_size * B}

    # ---- roofline ----
    if B == 1:
        # dominant kernel (rmsnorm + W1/W3 + SwiGLU) timed alone, layers cycled
        reps = max(1, 64 // wl.n_layers)
        dec.launch_op("w13", 0, 1)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for _ in range(reps):
            for layer in range(wl.n_layers):
                dec.launch_op("w13", layer, 1)
        k1.record(stream)
        k1.synchronize()
        w13_ms = k0.elapsed_time(k1) / (reps * wl.n_layers)
        achieved = w13_bytes(wl, wb) / (w13_ms / 1000.0) / 1e9
        traffic = None
        if (wl.dim, wl.hidden_dim) == (4096, 11008):
            src = open(os.path.join(ROOT, "llama_transformer_decode_gb300", "csrc", "gemv.cu"), "rb").read()
            nbytes, sources = W13_NCU_TRAFFIC["bf16" if bf16 else "f32"]
            if hashlib.sha256(src).hexdigest()[:16] in sources:
                traffic = nbytes
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": traffic,
                    "kernel": "l2dec_matvec_kernel<8,3,512,GEMV_W13> (rmsnorm + W1/W3 + SwiGLU)" + (", bf16 weights" if bf16 else ""),
                    "bytes_per_launch": w13_bytes(wl, wb), "us_per_launch": w13_ms * 1000.0,
                    "timing": "CUDA events around standalone launches on the decoder's stream, layers cycled",
                    "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                    # context, not the denominator: a pure read stream of the same 8 KB bulk copies
                    "read_ceiling": {"gbs": READ_CEILING_GBS, "frac": achieved / READ_CEILING_GBS,
                                     "source": "a 2 GiB read through per-warp rings of 8 KB 1-D bulk copies, nothing "
                                               "computed, measured on GB300 at 7.25-7.29 TB/s (the lower figure)"}}
    else:
        # whole batched step: B/2 flop per weight byte
        flops = 2.0 * B * (weight_bytes(wl) / 4.0) * args.steps  # 2 flops per weight (fp32 byte count / 4) per row
        tflops = flops / (ms / 1000.0) / 1e12
        alu = fp32_alu_peak_tflops(props)
        if on_tensor_cores(B, bf16):
            # tensor-core GEMV: 3 tf32 products per multiply-add are far below the tensor
            # peak, so the weights streamed from HBM bound it.  The dominant kernel (rmsnorm +
            # W1/W3 + SwiGLU) timed alone at this batch, layers cycled, as at batch 1.
            reps = max(1, 64 // wl.n_layers)
            dec.launch_op("w13", 0, 1, batch=B)
            k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            k0.record(stream)
            for _ in range(reps):
                for layer in range(wl.n_layers):
                    dec.launch_op("w13", layer, 1, batch=B)
            k1.record(stream)
            k1.synchronize()
            w13_ms = k0.elapsed_time(k1) / (reps * wl.n_layers)
            byts = w13_bytes(wl, wb) + 4 * (B - 1) * (wl.dim + wl.hidden_dim)  # B input and output rows
            achieved = byts / (w13_ms / 1000.0) / 1e9
            roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                        "traffic": None,
                        "kernel": "l2dec_matvec_tc_kernel<GEMV_W13> (rmsnorm + W1/W3 + SwiGLU, tensor cores, "
                                  f"{B} rows)" + (", bf16 weights" if bf16 else ""),
                        "bytes_per_launch": byts, "us_per_launch": w13_ms * 1000.0,
                        "timing": "CUDA events around standalone launches on the decoder's stream, layers cycled",
                        "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                        "step": {"achieved": step_gbs, "frac": step_gbs / hbm,
                                 "what": "whole batched step: weights + KV cache rows over the step time"}}
        elif B / 2.0 < alu * 1e3 / hbm:  # B/2 flop per weight byte, below the fp32 ridge point
            roofline = {"bound": "hbm", "achieved": step_gbs, "peak": hbm, "unit": "GB/s", "frac": step_gbs / hbm,
                        "traffic": None, "kernel": "whole batched step (all kernels)",
                        "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"}
        else:
            roofline = {"bound": "alu", "achieved": tflops, "peak": alu, "unit": "TFLOP/s", "frac": tflops / alu,
                        "traffic": None, "kernel": "whole batched step (all kernels)",
                        "peak_source": "fp32 FMA peak derived: SMs x 128 lanes x 2 flop x max SM clock"}
    dec.sync()

    # ---- CPU baseline: the oracle on this host's cores ----
    cpu = None
    if cpu_leg:
        n, el, threads = oracle_rate(wl, host_w, streams[0], args.cpu_budget)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} teacher-forced oracle steps of {wl.name} (one sequence) at positions 0..{n - 1}"}

    # ---- every workload's own rate (after the headline decoder is freed) ----
    per_config = None
    entries = parse_per_config(args.per_config) if (B == 1 and not bf16 and world == 1) else []
    if entries:
        dec.close()
        del w_dev
        dec = None
        per_config = per_config_rates(entries, hbm, peak_src, args.per_config_runs)

    clk = clocks.summary()
    cfg = config_of(wl, B, bf16)
    cfg["positions"] = (f"{timed_pos[0][0]}..{timed_pos[-1][0]}" if B == 1 else
                        f"slot b from floor(b*{S}/{B}) + {args.warmup}, {args.steps} steps, wrapping at {S}")
    metric = metric_of(B, bf16)
    if bf16:
        cfg["weights"] = "seeded random (synth); matrices streamed as bf16 (rounded once on the device), fp32 arithmetic"
    line = {
        "metric": metric,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded random weights and tokens)",
        "config": cfg,
        "hbm_roofline": {"achieved_gbs": step_gbs, "frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                         "frac_of_measured": step_gbs / hbm,
                         "bytes_per_step_avg": bytes_total / max(1, len(timed_pos))},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "per_position": per_pos or None,
        "per_config": per_config,
        "gpu_launches": kern * args.steps, "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    if dec is not None:
        dec.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_ours_prefill(args, wl):
    """A step is one l2_prefill of the T-token prompt from position 0 of slot 0
    (the slot rewound first): 64-row chunks, each a batched step."""
    import torch
    import torch.distributed as dist

    import llama_transformer_decode_gb300 as pkg

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    pkg._native.load()
    props = torch.cuda.get_device_properties(local_rank)
    T = args.prefill
    cpu_leg = rank == 0 and world == 1 and not args.no_cpu
    w_dev, host_w = load_weights_device(wl, keep_host=cpu_leg)
    stream = torch.cuda.Stream()
    dec = pkg.Decoder(wl.config_tuple(), w_dev, max_batch=1, stream=stream)
    toks = synth.token_stream(wl, 0, T)
    out = torch.empty((T, wl.vocab_size), device="cuda")
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs")
    peak_src = "of measured" if hbm else "of fallback"
    hbm = hbm or FALLBACK_HBM_GBS

    def step():
        dec.reset(0)
        dec.prefill(toks, pos0=0, slot=0, out=out)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    dec.sync()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(str(props.uuid)) as clocks:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    dec.sync()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    value = job_rate(T * args.steps, world, ms / 1000.0)

    # end to end: host tokens in (inside the call), the last row's logits back every step
    host_last = np.empty(wl.vocab_size, np.float32)
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
        stream.synchronize()
        host_last[:] = out[T - 1].cpu().numpy()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    dec.sync()
    e2e = {"value": job_rate(T * args.steps, world, e2e_s), "unit": "tokens/s",
           "h2d_bytes_per_step": dec.step_input_bytes() * len(prefill_chunks(T)),  # tokens ride in each chunk's block
           "d2h_bytes_per_step": 4 * wl.vocab_size}

    gbs = prefill_bytes(wl, T) * args.steps / (ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "traffic": None,
                "kernel": "whole prefill (all kernels of every chunk)",
                "bytes_per_step": prefill_bytes(wl, T),
                "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"}
    cpu = None
    if cpu_leg:
        n, el, threads = oracle_rate(wl, host_w, toks, args.cpu_budget)
        cpu = {"value": n / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"the first {n} tokens of the same prompt, teacher-forced one per oracle step"}
    launches = sum(5 * wl.n_layers + 1 + (1 if r >= TC_MIN_BATCH else 0) for _, r in prefill_chunks(T))
    cfg = config_of(wl, 1)
    cfg.update({"prefill_tokens": T, "chunk_rows": PREFILL_CHUNK, "positions": f"0..{T - 1}, slot rewound each step",
                "gemv": "tensor cores for chunks of 16+ rows (tcgen05 kind::tf32, 3-term hi/lo split), "
                        "CUDA cores below"})
    clk = clocks.summary()
    line = {
        "metric": metric_of(1, prefill=T), "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded random weights and tokens)",
        "config": cfg, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches * args.steps, "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    dec.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: to the end of the context)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="llama2_7b", choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=1,
                    help="independent sequences per step at staggered positions (batched_1b: 16 or 64)")
    ap.add_argument("--weights", choices=("f32", "bf16"), default="f32",
                    help="bf16: matrices streamed as bf16 (L2_FLAG_BF16_WEIGHTS)")
    ap.add_argument("--prefill", type=int, default=0, metavar="T",
                    help="time l2_prefill of a T-token prompt instead of decode steps (one prompt per step)")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode only the first N layers of the workload (a smaller case, e.g. for profiling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-positions", action="store_true", help="skip the per-position rates")
    ap.add_argument("--per-config", default=None, metavar="LIST",
                    help="workloads whose own rates the batch-1 decode line reports, as name[:batch],... "
                         f"(default for llama2_7b: {DEFAULT_PER_CONFIG}; 'none' skips)")
    ap.add_argument("--per-config-runs", type=int, default=5, help="timed runs per entry of --per-config (median)")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--reference-budget", type=float, default=90.0,
                    help="seconds of timed oracle work in --impl reference")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if not 1 <= args.batch <= 64:
        ap.error("--batch must be in 1..64")
    if args.weights == "bf16" and args.impl != "ours":
        ap.error("--weights bf16 is an option of this implementation, not of the reference arm")
    if args.per_config is None:
        args.per_config = DEFAULT_PER_CONFIG if args.workload == "llama2_7b" and args.layers is None else "none"
    try:
        parse_per_config(args.per_config)
    except ValueError as e:
        ap.error(str(e))
    if args.per_config_runs < 1:
        ap.error("--per-config-runs must be at least 1")
    wl = WORKLOADS[args.workload]
    if args.layers is not None:
        if not 1 <= args.layers <= wl.n_layers:
            ap.error(f"--layers must be in 1..{wl.n_layers}")
        wl = wl.replace(n_layers=args.layers, name=f"{wl.name} ({args.layers} layers)")
    if args.prefill:
        if not 1 <= args.prefill <= wl.seq_len:
            ap.error(f"--prefill must be in 1..{wl.seq_len}")
        if args.batch != 1 or args.weights != "f32":
            ap.error("--prefill times one prompt with fp32 weights")
        if args.steps is None:
            args.steps = 5
    if args.steps is None:
        args.steps = max(1, wl.seq_len - args.warmup)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours_prefill(args, wl) if args.prefill else run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
