#!/usr/bin/env python
"""Benchmark of the verify step (kv_append_quant -> verify_attn -> spec_accept).

Default workload: 8 lanes with contexts uniform in [4096, 65536], 24 q / 4 kv
heads, head_dim 128, window 1 + 15 drafts, FP8 E4M3 KV (page 64, permuted page
table), acceptance over a 151,936-token vocabulary.  Inputs are seeded and
synthetic and already resident in HBM when the timed region starts.

One JSON line (rank 0):
  value        verify steps/s (verify_step: append + verify_attn + spec_accept
               as one chain of programmatic dependent launches), device time
  verify_attn  achieved algorithmic HBM GB/s of the verify_attn call and its
               fraction of the measured copy bandwidth (roofline object)
  e2e          the same steps/s through the C ABI from pinned HOST buffers,
               host->device inputs and device->host results inside the timing
               (the logits copy overlaps append and verify: only accept reads it,
               lane chunk by lane chunk as the chunks land)
  cpu_baseline the CPU oracle on the host cores, on a bounded sample
  spec_accept_lazy  the acceptance that reads each lane's logits rows only up
               to its first disagreement (timed apart, after the main loop),
               with the step rate it would give
  spec_accept_sampled  lossless stochastic acceptance with a synthetic draft
               distribution (timed apart likewise)
  all_workloads every workload's verify_attn time, GB/s and fraction of the
               measured peak, and its step time, measured the same way
  clocks       nvidia-smi SM clocks and throttle reasons during the timed steps

Timing: W untimed warm-up steps, then K steps, each preceded by an untimed L2
flush (a 512 MB write, then a 512 MB read of a second buffer, so that L2 holds
none of the step's inputs and none of the write's dirty lines), each bracketed
by CUDA events on the launching stream; a barrier and a device synchronize
bracket the whole timed loop.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
Multi-GPU: torchrun, one replica per GPU (lanes are independent: no collective).
"""
from __future__ import annotations

import argparse
import json
import math
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

SM_SCALE = np.float32(1.0 / math.sqrt(128.0))
METRIC = "verify_attn HBM GB/s (% of GB300 peak) and verify steps/s at 8 lanes"
DEFAULT_WORKLOAD = "multi_lane"
# dram bytes (read + write) of one verify_attn call (split + merge kernels),
# from an ncu capture of the kernels built from sources with this SHA-256
# (verify_attn_tc.cu, tc_primitives.cuh, verify_attn.cu, in that order, comments stripped);
# reported as null once the sources differ (the counters are then stale).
NCU_TRAFFIC = {"sources_sha256": "44309ab667511223cc8f80338fd680afc3acd8be96ad613058a6664407bfaf02",
               "bytes": {"multi_lane": 314707456, "long_context": 249022464, "int4_12slot": 338031360,
                         "multi_lane_int8": 324021760, "multi_lane_fp8row": 323727872}}
TRAFFIC_SOURCES = ("verify_attn_tc.cu", "tc_primitives.cuh", "verify_attn.cu")


def code_of(text: str) -> str:
    """A source file without its // comments, trailing blanks and empty lines:
    what the counters depend on (the files hold no block comments and no //
    inside string literals)."""
    lines = (ln.split("//", 1)[0].rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for n in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "speculative_decode_verify_append_gb300", "csrc", n), encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()


def ncu_traffic(name: str):
    if NCU_TRAFFIC["sources_sha256"] != kernel_sources_sha256():
        return None
    return NCU_TRAFFIC["bytes"].get(name)


def workload_desc(spec: synth.Spec) -> str:
    kv = {synth.KV_FP8: "FP8 E4M3 KV, fp32 scale per (page, head)",
          synth.KV_INT4: "INT4 KV, fp16 scale per group of 32",
          synth.KV_INT8: "INT8 KV, fp16 scale per group of 64",
          synth.KV_FP8_ROW: "FP8 E4M3 KV, fp32 scale per (token, head) row"}[spec.kv_dtype]
    ctx = f"context {spec.ctx_lo}" if spec.ctx_lo == spec.ctx_hi else f"contexts U[{spec.ctx_lo}, {spec.ctx_hi}]"
    acc = f", acceptance over vocab {spec.vocab} (p={spec.match_p})" if spec.vocab else ""
    return (f"{spec.name}: {spec.num_lanes} lanes, {ctx}, {spec.num_q_heads} q / {spec.num_kv_heads} kv heads, "
            f"head_dim 128, window 1+{spec.window - 1}, {kv}, page 64, "
            f"{'permuted' if spec.permuted else 'identity'} page table{acc}")


def verify_algorithmic_bytes(spec: synth.Spec, seq_lens: np.ndarray) -> int:
    """HBM bytes verify_attn must move at minimum: every visible key's K and V
    codes and scales once, Q in, O out, the page-table entries used."""
    W, Hq, Hkv = spec.window, spec.num_q_heads, spec.num_kv_heads
    tokens = int(np.sum(seq_lens.astype(np.int64) + W))
    pages = int(np.sum((seq_lens.astype(np.int64) + W + 63) // 64))
    if spec.kv_dtype == synth.KV_FP8:
        kv = tokens * Hkv * 256 + pages * Hkv * 8          # E4M3 codes; fp32 K and V scale per page
    elif spec.kv_dtype == synth.KV_INT4:
        kv = tokens * Hkv * (128 + 16)                      # nibbles; 4 fp16 scales each for K and V
    elif spec.kv_dtype == synth.KV_INT8:
        kv = tokens * Hkv * (256 + 8)                       # int8 codes; 2 fp16 scales each for K and V
    else:
        kv = tokens * Hkv * (256 + 8)                       # E4M3 codes; one fp32 scale each for K and V
    qo = 2 * len(seq_lens) * W * Hq * 128 * 2
    return kv + qo + pages * 4 + len(seq_lens) * 4


KV_LABELS = {synth.KV_FP8: "fp8", synth.KV_INT4: "int4", synth.KV_INT8: "int8-g64", synth.KV_FP8_ROW: "fp8-row"}


def all_workload_specs() -> dict:
    """Every workload, plus the 8-lane workload in the INT8 group-64 and FP8
    row-scale cache formats (same lengths, values and shapes)."""
    import dataclasses
    specs = dict(synth.WORKLOADS)
    base = synth.WORKLOADS["multi_lane"]
    for dt, tag in ((synth.KV_INT8, "int8"), (synth.KV_FP8_ROW, "fp8row")):
        specs[f"multi_lane_{tag}"] = dataclasses.replace(base, name=f"multi_lane_{tag}", kv_dtype=dt)
    return specs


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# shared by both arms
# ---------------------------------------------------------------------------
def bench_config(spec: synth.Spec, seq_lens: np.ndarray, world: int) -> dict:
    """The `config` object of the JSON line (identical in both arms)."""
    return {"workload": workload_desc(spec), "lanes": int(len(seq_lens)), "window": spec.window,
            "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads, "context_tokens": int(seq_lens.sum()),
            "parallelism": f"replicas x{world}",
            "l2": "flushed before every timed step (512 MB write, then 512 MB read of a second buffer; untimed)"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_setup(spec: synth.Spec, step: synth.Step, lanes):
    import oracle
    cache = oracle.Cache(spec.kv_dtype, step.num_pages, spec.num_kv_heads)
    for b in lanes:
        for start, n in synth.fill_chunks(int(step.seq_lens[b])):
            k, v = synth.context_chunk(spec, b, start, n)
            oracle.append(cache, k[None], v[None], step.page_table[b:b + 1], np.array([start], np.int32))
    return cache


def lane_work(spec: synth.Spec, L: int) -> float:
    """Attention work of one lane's window (rows x visible keys)."""
    W = spec.window
    return W * spec.num_q_heads * (int(L) + (W + 1) / 2)


def oracle_lane_step(step: synth.Step, cache, b: int, threads: int) -> float:
    """One lane's whole verify step on the CPU oracle -- the window append,
    every window row's attention in fp64, the acceptance -- in seconds.  The
    append rewrites the same slots with the same values each time."""
    import oracle
    B, W, Hq = step.q.shape[:3]
    sel = slice(b, b + 1)
    t0 = time.perf_counter()
    oracle.append(cache, step.k_win[sel], step.v_win[sel], step.page_table[sel], step.seq_lens[sel])
    rows = [(b, i, h) for i in range(W) for h in range(Hq)]
    oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM_SCALE, rows=rows, threads=threads)
    if step.logits is not None:
        oracle.spec_accept(step.logits[sel], step.drafts[sel], step.seq_lens[sel])
    return time.perf_counter() - t0


def oracle_steps(spec, step, cache, lanes, threads, n_steps=None, budget_s=None):
    """Lane-steps cycling over `lanes` (n_steps of them, or until budget_s has
    passed and every lane ran once).  Returns (seconds per timed lane-step,
    full-workload steps per second, lane-steps run)."""
    times, work = [], 0.0
    full = sum(lane_work(spec, L) for L in step.seq_lens)
    t_start = time.perf_counter()
    k = 0
    while True:
        if n_steps is not None and k >= n_steps:
            break
        if budget_s is not None and k >= len(lanes) and time.perf_counter() - t_start > budget_s:
            break
        b = lanes[k % len(lanes)]
        times.append(oracle_lane_step(step, cache, b, threads))
        work += lane_work(spec, step.seq_lens[b])
        k += 1
    total = float(np.sum(times))
    return total / max(1, len(times)), (work / full) / total, len(times)


REFERENCE_BUDGET_S = 120.0  # host time the reference arm's warm-up and timed steps aim at together


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, sized by a
    calibration so that the W + K steps take about REFERENCE_BUDGET_S
    together, whatever W and K are.  When a step's share allows at least one
    wave of rows over all threads, a step is a run of consecutive attention
    rows of the workload (lane by lane, window position by position, head by
    head, cycling), each lane's window append and acceptance done in the step
    that reaches its first and last row; otherwise a step is one row over as
    many of its keys as its share allows, on one thread.  `value` counts the
    keys attended in whole-workload steps per second."""
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    spec = all_workload_specs()[args.workload]
    step = synth.make_step(spec)
    B, W, Hq = step.q.shape[:3]
    lanes = list(range(B))
    cache = oracle_setup(spec, step, lanes)
    threads = os.cpu_count() or 1
    rows_all = [(b, i, h) for b in lanes for i in range(W) for h in range(Hq)]
    full = sum(lane_work(spec, L) for L in step.seq_lens)
    per_step = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    # calibration on the median lane: one wave of `threads` rows in parallel
    bm = int(np.argsort(step.seq_lens)[len(lanes) // 2])
    wave = [(bm, i, h) for i in range(W) for h in range(Hq)][:max(1, min(threads, W * Hq))]
    t0 = time.perf_counter()
    oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM_SCALE, rows=wave, threads=threads)
    t_wave = time.perf_counter() - t0
    row_mode = per_step >= t_wave
    if row_mode:
        # whole rows: a multiple of the thread count, at most one lane's window
        rows_per_step = int(min(W * Hq, len(wave) * max(1, int(per_step // t_wave))))
        cores = min(threads, rows_per_step)
    else:
        # a step shorter than one wave of rows: one row over the first n_keys of its keys, on one thread
        L0 = int(step.seq_lens[bm])
        t0 = time.perf_counter()
        oracle.decode_row(cache, step.q[bm, 0, 0], 0, step.page_table[bm], L0 + 1, SM_SCALE)
        sec_per_key = (time.perf_counter() - t0) / (L0 + 1)
        rows_per_step = 1
        cores = 1
    pos = 0

    def one_step():
        nonlocal pos
        if not row_mode:
            b, i, h = rows_all[pos % len(rows_all)]
            pos = (pos + 1) % len(rows_all)
            n_keys = int(max(1, min(int(step.seq_lens[b]) + i + 1, per_step / max(sec_per_key, 1e-12))))
            t1 = time.perf_counter()
            oracle.decode_row(cache, step.q[b, i, h], h // (Hq // spec.num_kv_heads), step.page_table[b], n_keys,
                              SM_SCALE)
            return time.perf_counter() - t1, n_keys
        rows = [rows_all[(pos + k) % len(rows_all)] for k in range(rows_per_step)]
        pos = (pos + rows_per_step) % len(rows_all)
        t1 = time.perf_counter()
        for (b, i, h) in rows:
            if i == 0 and h == 0:  # the lane's append precedes its attention
                sel = slice(b, b + 1)
                oracle.append(cache, step.k_win[sel], step.v_win[sel], step.page_table[sel], step.seq_lens[sel])
        oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM_SCALE, rows=rows, threads=threads)
        for (b, i, h) in rows:
            if i == W - 1 and h == Hq - 1 and step.logits is not None:  # the lane's acceptance
                sel = slice(b, b + 1)
                oracle.spec_accept(step.logits[sel], step.drafts[sel], step.seq_lens[sel])
        dt = time.perf_counter() - t1
        return dt, sum(int(step.seq_lens[b]) + i + 1 for (b, i, h) in rows)

    for _ in range(args.warmup):
        one_step()
    times, work = [], 0
    for _ in range(args.steps):
        dt, wk = one_step()
        times.append(dt)
        work += wk
    total = float(np.sum(times))
    value = (work / full) / total if total > 0 else 0.0
    model = cpu_model()
    if row_mode:
        unit = f"{rows_per_step} attention rows per timed step"
        sample = (f"each step: {rows_per_step} consecutive attention rows of the {B}-lane workload (of "
                  f"{len(rows_all)}), cycling over lanes, window positions and heads, over each row's whole "
                  f"context in fp64 ({cores} threads), a lane's window append and acceptance in the step that "
                  f"reaches its first and last row")
    else:
        unit = "one attention row over a bounded number of its keys per timed step"
        sample = (f"each step: one attention row of the {B}-lane workload, cycling over lanes, window positions "
                  f"and heads, over its first keys (as many as the step's share of the budget allows), fp64 on "
                  f"one thread")
    sample += (f"; sized so that {args.warmup} + {args.steps} steps take about {REFERENCE_BUDGET_S:.0f} s; "
               f"value = whole-workload steps/s of the keys attended")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / max(1, args.steps) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": bench_config(spec, step.seq_lens, world),
        "step_unit": f"{unit} (see cpu_baseline.sample)",
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "kind": "oracle", "cpu": model,
                         "sample": sample},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
class GpuWorkload:
    """One workload resident on the device: the cache filled by the library's
    own append, the step's inputs, the per-shape buffers."""

    def __init__(self, spec: synth.Spec, dev):
        import torch

        import speculative_decode_verify_append_gb300 as sdva
        from speculative_decode_verify_append_gb300.step import VerifyStep, fill_context
        self.spec = spec
        self.step = step = synth.make_step(spec)
        B, W, Hq = step.q.shape[:3]
        Hkv = spec.num_kv_heads

        def bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        self.cache = sdva.KVCache(spec.kv_dtype, step.num_pages, Hkv, device=dev)
        self.table = torch.from_numpy(step.page_table).to(dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        for b in range(B):
            L = int(step.seq_lens[b])
            for start, n in synth.fill_chunks(L, 16384):
                k, v = synth.context_chunk(spec, b, start, n)
                fill_context(self.cache, bf16(k), bf16(v), self.table[b], start=start, chunk=4096, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        self.seq = torch.from_numpy(step.seq_lens).to(dev)
        self.commit_lens = self.seq.clone()  # the commit advances a copy: every timed step does the same work
        self.q, self.kw, self.vw = bf16(step.q), bf16(step.k_win), bf16(step.v_win)
        self.logits = torch.from_numpy(step.logits).to(dev) if step.logits is not None else None
        self.drafts = torch.from_numpy(step.drafts).to(dev) if step.drafts is not None else None
        self.vs = VerifyStep(B, W, Hq, Hkv, spec.ctx_hi, spec.vocab, device=dev)
        self.alg = verify_algorithmic_bytes(spec, step.seq_lens)

    def separate(self, evs=None):
        """append, verify_attn, spec_accept as three calls; events between them."""
        import torch
        stream = torch.cuda.current_stream()
        if evs:
            evs[0].record(stream)
        self.vs.append(self.cache, self.kw, self.vw, self.table, self.seq)
        if evs:
            evs[1].record(stream)
        self.vs.attend(self.cache, self.q, self.table, self.seq)
        if evs:
            evs[2].record(stream)
        if self.logits is not None:
            self.vs.accept(self.logits, self.drafts, self.commit_lens)
        if evs:
            evs[3].record(stream)

    def reset(self):
        """Before a chained step (untimed): the step commits into commit_lens,
        which starts every step at the pre-step lengths, so that every timed
        step repeats the same work."""
        self.commit_lens.copy_(self.seq)

    def chained(self):
        """The whole step in one call (verify_step), or append + verify when the
        workload has no acceptance."""
        if self.logits is None:
            self.separate()
            return
        self.vs.step(self.cache, self.q, self.kw, self.vw, self.table, self.commit_lens, self.logits, self.drafts,
                     commit=True)

    def launches_per_step(self) -> int:
        return 3 + (2 if self.logits is not None else 0)


def time_loop(fn, n_steps, n_warmup, flush_l2, n_events=2):
    """n_warmup untimed then n_steps timed calls of fn(evs), each after an L2
    flush; returns the per-step event lists."""
    import torch
    for _ in range(n_warmup):
        flush_l2()
        fn(None)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_events)] for _ in range(n_steps)]
    for k in range(n_steps):
        flush_l2()
        fn(evs[k])
    torch.cuda.synchronize()
    return evs


def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import speculative_decode_verify_append_gb300 as sdva

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        # The write evicts the step's inputs; the read of a second buffer then
        # evicts the write's dirty lines, whose write-back would otherwise land
        # inside the timed step.
        flush.zero_()
        clean.amax()
    stream = torch.cuda.current_stream()

    spec = all_workload_specs()[args.workload]
    wl = GpuWorkload(spec, dev)
    step, vs = wl.step, wl.vs
    B, W, Hq = step.q.shape[:3]
    logits, drafts = wl.logits, wl.drafts

    # ---- the timed steps: verify_step, one call per step ----
    def chained_step(evs, w=wl):
        w.reset()
        if evs:
            evs[0].record(stream)
        w.chained()
        if evs:
            evs[1].record(stream)
    for _ in range(args.warmup):
        flush_l2()
        chained_step(None)
    torch.cuda.synchronize()
    assert int(vs.status.item()) == 0, sdva.sdva_status_string(int(vs.status.item()))

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler see the GPU under load from the first step
    wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed_steps")
    for k in range(args.steps):
        flush_l2()
        chained_step(evs[k])
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(dist)
    clocks = sampler.stop()
    assert int(vs.status.item()) == 0, sdva.sdva_status_string(int(vs.status.item()))
    t_step = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = max_over_ranks(dist, float(np.sum(t_step)))
    ms_per_step = total_ms / args.steps
    value = world * args.steps / (total_ms / 1e3)

    # ---- the same step as three calls, timed apart: the per-call breakdown ----
    sep = time_loop(wl.separate, args.steps, args.warmup, flush_l2, 4)
    t_app = [e[0].elapsed_time(e[1]) for e in sep]
    t_att = [e[1].elapsed_time(e[2]) for e in sep]
    t_acc = [e[2].elapsed_time(e[3]) for e in sep]
    t_sep = [e[0].elapsed_time(e[3]) for e in sep]

    # ---- lazy acceptance (rows read only up to each lane's first disagreement) ----
    lazy = None
    if logits is not None:
        l_ev = time_loop(lambda e: (e and e[0].record(stream), vs.accept_lazy(logits, drafts, None, wl.commit_lens),
                                    e and e[1].record(stream)), args.steps, args.warmup, flush_l2)
        acc_lazy = vs.accept_len.cpu().numpy().copy()
        tok_lazy = vs.out_tokens.cpu().numpy().copy()
        vs.accept(logits, drafts, None)
        torch.cuda.synchronize()
        acc_eager, tok_eager = vs.accept_len.cpu().numpy(), vs.out_tokens.cpu().numpy()
        assert np.array_equal(acc_lazy, acc_eager), (acc_lazy, acc_eager)
        for b in range(B):
            assert np.array_equal(tok_lazy[b, :acc_lazy[b] + 1], tok_eager[b, :acc_lazy[b] + 1])
        assert int(vs.status.item()) == 0, sdva.sdva_status_string(int(vs.status.item()))
        t_lazy = float(np.mean([e[0].elapsed_time(e[1]) for e in l_ev]))
        walk = B >= sdva.LAZY_WALK_MIN_LANES
        rows_needed = int((1 + acc_lazy).sum())
        rows_read = rows_needed if walk else B * W
        lazy_bytes = rows_read * spec.vocab * 4 + B * (W - 1) * 4
        lazy_step_us = (float(np.mean(t_app)) + float(np.mean(t_att)) + t_lazy) * 1e3
        lazy = {"us": t_lazy * 1e3, "mode": "walk" if walk else "parallel", "rows_needed": rows_needed,
                "rows_read": rows_read, "rows_in_window": B * W, "accept_len": [int(a) for a in acc_lazy],
                "bytes_read": lazy_bytes, "gbs": lazy_bytes / (t_lazy / 1e3) / 1e9,
                "eager_us": float(np.mean(t_acc)) * 1e3, "step_us": lazy_step_us, "steps_per_s": 1e6 / lazy_step_us,
                "timing": "CUDA events around the call after an L2 flush, same steps and warm-up as the main loop"}

    # ---- lossless stochastic acceptance with the draft distribution q ----
    sampled = None
    if logits is not None:
        gen = torch.Generator(device=dev)
        gen.manual_seed(spec.seed)
        # a draft distribution correlated with the target, drafts drawn from it
        zq = 0.8 * logits[:, :W - 1] + 0.6 * torch.randn(logits[:, :W - 1].shape, generator=gen, device=dev)
        qd = torch.softmax(zq, dim=2).contiguous()
        del zq
        dq = torch.multinomial(qd.view(-1, spec.vocab), 1, generator=gen).view(B, W - 1).to(torch.int32).contiguous()
        ua = torch.rand((B, W - 1), generator=gen, device=dev)
        us = torch.rand(B, generator=gen, device=dev)
        ws = torch.empty(sdva.spec_accept_sampled_workspace_size(B, W), dtype=torch.uint8, device=dev)
        s_acc = torch.zeros(B, dtype=torch.int32, device=dev)
        s_tok = torch.zeros((B, W), dtype=torch.int32, device=dev)
        s_ev = time_loop(lambda e: (e and e[0].record(stream),
                                    sdva.spec_accept_sampled(logits, qd, dq, ua, us, s_acc, s_tok, ws, wl.commit_lens,
                                                             vs.status),
                                    e and e[1].record(stream)), args.steps, args.warmup, flush_l2)
        assert int(vs.status.item()) == 0, sdva.sdva_status_string(int(vs.status.item()))
        t_s = float(np.mean([e[0].elapsed_time(e[1]) for e in s_ev]))
        a_s = s_acc.cpu().numpy()
        # every logits row for the statistics, then per lane the drawn row and,
        # after a rejection, its draft row; one logit and one q entry per tested draft
        s_bytes = (B * W * spec.vocab * 4 + B * spec.vocab * 4 + int((a_s < W - 1).sum()) * spec.vocab * 4
                   + int(np.minimum(a_s + 1, W - 1).sum()) * 16)
        s_step_us = (float(np.mean(t_app)) + float(np.mean(t_att)) + t_s) * 1e3
        sampled = {"us": t_s * 1e3, "accept_len": [int(a) for a in a_s], "bytes_read": s_bytes,
                   "gbs": s_bytes / (t_s / 1e3) / 1e9, "step_us": s_step_us, "steps_per_s": 1e6 / s_step_us,
                   "inputs": "q = softmax(0.8 * target logits + 0.6 * N(0,1)), drafts drawn from q, uniforms "
                             "from a seeded device generator",
                   "timing": "CUDA events around the call after an L2 flush, same steps and warm-up as the main loop"}
        del qd

    # ---- the attention's other modes on the same workload: per-lane row counts, a draft tree ----
    modes = None
    if not args.no_all_workloads:
        rng = np.random.default_rng(11)
        counts = rng.integers(1, W + 1, size=B).astype(np.int32)
        parent = np.zeros((B, W), np.int32)
        for i in range(1, W):
            parent[:, i] = rng.integers(0, i, size=B)
        n_dev = torch.from_numpy(counts).to(dev)
        full_dev = torch.full((B,), W, dtype=torch.int32, device=dev)
        par_dev = torch.from_numpy(parent).to(dev)
        mc = spec.ctx_hi

        def timed(call):
            def fn(e):
                if e:
                    e[0].record(stream)
                call()
                if e:
                    e[1].record(stream)
            evs = time_loop(fn, args.steps, args.warmup, flush_l2)
            return 1e3 * float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
        ws = vs.workspace
        t_causal = timed(lambda: sdva.verify_attn(wl.cache, wl.q, wl.table, wl.seq, mc, float(SM_SCALE), vs.out, ws,
                                                  vs.status))
        t_full = timed(lambda: sdva.verify_attn_ragged(wl.cache, wl.q, full_dev, wl.table, wl.seq, mc, float(SM_SCALE),
                                                       vs.out, ws, vs.status))
        t_rag = timed(lambda: sdva.verify_attn_ragged(wl.cache, wl.q, n_dev, wl.table, wl.seq, mc, float(SM_SCALE),
                                                      vs.out, ws, vs.status))
        t_tree = timed(lambda: sdva.verify_attn_tree(wl.cache, wl.q, par_dev, wl.table, wl.seq, mc, float(SM_SCALE),
                                                     vs.out, ws, vs.status))
        assert int(vs.status.item()) == 0, sdva.sdva_status_string(int(vs.status.item()))
        modes = {"verify_attn_us": t_causal, "verify_attn_ragged_full_counts_us": t_full,
                 "verify_attn_ragged_us": t_rag, "ragged_counts": [int(c) for c in counts],
                 "ragged_rows_fraction": float(counts.sum()) / (B * W), "verify_attn_tree_us": t_tree,
                 "tree": "random: slot i hangs under a uniform earlier slot (seed 11)",
                 "timing": "CUDA events around the call after an L2 flush, same steps and warm-up as the main loop"}

    # ---- e2e: host buffers through the public API ----
    q, kw, vw, seq, table, cache = wl.q, wl.kw, wl.vw, wl.seq, wl.table, wl.cache
    host_in = {n: t.cpu().pin_memory() for n, t in (("q", q), ("kw", kw), ("vw", vw))}
    if logits is not None:
        host_in["logits"] = logits.cpu().pin_memory()
        host_in["drafts"] = drafts.cpu().pin_memory()
    host_out = {"out": torch.empty_like(vs.out, device="cpu").pin_memory(),
                "acc": torch.empty_like(vs.accept_len, device="cpu").pin_memory(),
                "tok": torch.empty_like(vs.out_tokens, device="cpu").pin_memory()}
    dev_in = {"q": q, "kw": kw, "vw": vw, "logits": logits, "drafts": drafts}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values()) if logits is not None else \
        host_out["out"].numel() * 2
    e2e_steps = max(10, min(args.steps, 200))
    e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    # The logits (most of a step's input bytes) are read only by spec_accept:
    # they are copied in two lane chunks on one side stream while append and
    # verify run, and each chunk's acceptance runs as soon as that chunk has
    # landed (lanes are independent), so only the last chunk's acceptance
    # follows the copy.  The attention output is read back on a second side
    # stream once verify_attn is done.  (The host link carried ~209 GB/s on
    # this part whether one copy, several concurrent copies or a kernel read
    # the pinned buffer.)  The step -- every copy and every call -- is captured
    # once in a CUDA graph and replayed each step, as a serving loop does: the
    # Python launch overhead of ~30 calls per step would otherwise leave the
    # GPU idle between them.
    cs = torch.cuda.Stream(device=dev)  # host -> device: logits
    ds = torch.cuda.Stream(device=dev)  # device -> host: attention output
    n_chunks = min(B, 2) if logits is not None else 0
    bounds = [(B * i // n_chunks, B * (i + 1) // n_chunks) for i in range(n_chunks)]

    def e2e_body():
        cur = torch.cuda.current_stream()
        ready = []
        # the small inputs first, so that append and verify do not wait behind the logits on the copy engine
        for n, t in host_in.items():
            if n != "logits":
                dev_in[n].copy_(t, non_blocking=True)
        if logits is not None:
            cs.wait_stream(cur)  # the previous step's acceptance has read the old logits
            with torch.cuda.stream(cs):
                for lo, hi in bounds:
                    dev_in["logits"][lo:hi].copy_(host_in["logits"][lo:hi], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                    ready.append(ev)
        vs.append(cache, kw, vw, table, seq)
        vs.attend(cache, q, table, seq)
        ds.wait_stream(cur)
        with torch.cuda.stream(ds):
            host_out["out"].copy_(vs.out, non_blocking=True)
        if logits is not None:
            for (lo, hi), ev in zip(bounds, ready):
                cur.wait_event(ev)
                sdva.spec_accept(logits[lo:hi], drafts[lo:hi], vs.accept_len[lo:hi], vs.out_tokens[lo:hi],
                                 wl.commit_lens[lo:hi], vs.status)
            host_out["acc"].copy_(vs.accept_len, non_blocking=True)
            host_out["tok"].copy_(vs.out_tokens, non_blocking=True)
        cur.wait_stream(ds)

    e2e_body()  # eager once (the library sets its per-device attributes outside the capture)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        e2e_body()
    torch.cuda.synchronize()
    for k in range(e2e_steps + 3):
        flush_l2()
        if k >= 3:
            e_ev[k - 3][0].record(stream)
        graph.replay()
        if k >= 3:
            e_ev[k - 3][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, float(np.sum([e[0].elapsed_time(e[1]) for e in e_ev])))
    e2e_value = world * e2e_steps / (e2e_ms / 1e3)

    # ---- roofline of the verify_attn call ----
    alg = wl.alg
    att_ms = float(np.mean(t_att))
    achieved = alg / (att_ms / 1e3) / 1e9
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]
    traffic = ncu_traffic(spec.name)

    # ---- every workload, same method: verify_attn alone and the whole step ----
    all_workloads = None
    if not args.no_all_workloads:
        all_workloads = {}
        for name, wspec in all_workload_specs().items():
            w = wl if name == spec.name else GpuWorkload(wspec, dev)
            e_sep = time_loop(w.separate, args.steps, args.warmup, flush_l2, 4)
            e_ch = time_loop(lambda e: chained_step(e, w), args.steps, args.warmup, flush_l2)
            assert int(w.vs.status.item()) == 0, (name, sdva.sdva_status_string(int(w.vs.status.item())))
            v_us = 1e3 * float(np.mean([e[1].elapsed_time(e[2]) for e in e_sep]))
            st_us = 1e3 * float(np.mean([e[0].elapsed_time(e[1]) for e in e_ch]))
            sep_us = 1e3 * float(np.mean([e[0].elapsed_time(e[3]) for e in e_sep]))
            gbs = w.alg / (v_us / 1e6) / 1e9
            all_workloads[name] = {"verify_attn_us": v_us, "verify_attn_gbs": gbs, "frac": gbs / peak,
                                   "algorithmic_bytes": w.alg, "traffic": ncu_traffic(name),
                                   "step_us": st_us, "steps_per_s": 1e6 / st_us,
                                   "separate_calls_step_us": sep_us, "kv": KV_LABELS[w.spec.kv_dtype]}
            if w is not wl:
                del w
                torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8-e4m3 KV (int4 for the 4-bit workload; int8 / fp8-row variants in all_workloads) -> "
                 "f16 tensor-core MMA, f32 accumulate, bf16 out",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, N(0,1) fp32 logits)",
        "config": bench_config(spec, step.seq_lens, world),
        "step": "verify_step: kv_append_quant + verify_attn + spec_accept as one chain of programmatic dependent "
                "launches",
        "verify_attn": {"us": att_ms * 1e3, "gbs": achieved, "pct_of_peak": 100.0 * achieved / peak,
                        "algorithmic_bytes": alg},
        "breakdown_us": {"kv_append_quant": float(np.mean(t_app)) * 1e3, "verify_attn": att_ms * 1e3,
                         "spec_accept": float(np.mean(t_acc)) * 1e3,
                         "three_separate_calls": float(np.mean(t_sep)) * 1e3,
                         "verify_step": ms_per_step * 1e3},
        "roofline": {"kernel": "verify_attn (split-K + merge kernels)", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic, "algorithmic_bytes": alg},
        "e2e": {"value": e2e_value, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "calls": "kv_append_quant, verify_attn, spec_accept and every host<->device copy of the step, "
                         "from pinned host buffers, captured once in a CUDA graph and replayed each step (the "
                         "logits copied in two lane chunks under append and verify, each chunk accepted as it "
                         "lands)"},
        "all_workloads": all_workloads,
        "spec_accept_lazy": lazy,
        "spec_accept_sampled": sampled,
        "verify_modes": modes,
        "gpu_launches": args.steps * wl.launches_per_step(),
        "clocks": clocks,
        "wall_s_timed_loop": wall,
    }

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        lanes = list(range(B))
        ocache = oracle_setup(spec, step, lanes)
        threads = os.cpu_count() or 1
        sec, cvalue, n = oracle_steps(spec, step, ocache, lanes, threads, budget_s=15.0)
        line["cpu_baseline"] = {
            "value": cvalue, "unit": "steps/s", "cores": threads, "kind": "oracle", "cpu": cpu_model(),
            "sample": f"{n} lane-steps cycling over the {B} lanes, each one lane's window append, all "
                      f"{W} x {Hq} attention rows over its whole context in fp64 ({threads} threads) and its "
                      f"acceptance; value = whole-workload steps/s of the work done"}
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_lazy_sweep(args):
    """Eager vs lazy acceptance over lane counts: 151,936 fp32 logits per row,
    16 positions, drafts agreeing with the argmax with probability 0.7 (seeded
    device RNG), L2 flushed before every call; one JSON line of mean us."""
    import torch

    import speculative_decode_verify_append_gb300 as sdva
    dev = torch.device("cuda", 0)
    V, W, p = 151936, 16, 0.7
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    res = {}
    for B in (8, 16, 32, 48, 64, 128):
        logits = torch.randn((B, W, V), generator=gen, device=dev)
        t = logits.argmax(dim=2).to(torch.int32)
        agree = torch.rand((B, W - 1), generator=gen, device=dev) < p
        drafts = torch.where(agree, t[:, :W - 1], (t[:, :W - 1] + 1) % V).to(torch.int32).contiguous()
        acc = torch.zeros(B, dtype=torch.int32, device=dev)
        tok = torch.zeros((B, W), dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        row = {}
        for name, fn in (("eager_us", lambda: sdva.spec_accept(logits, drafts, acc, tok, None, st)),
                         ("lazy_us", lambda: sdva.spec_accept_lazy(logits, drafts, acc, tok, None, None, st))):
            evs = []
            for k in range(args.warmup + args.steps):
                flush.zero_()
                clean.amax()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                if k >= args.warmup:
                    evs.append((e0, e1))
            torch.cuda.synchronize()
            row[name] = 1e3 * float(np.mean([a.elapsed_time(b) for a, b in evs]))
        assert int(st.item()) == 0, sdva.sdva_status_string(int(st.item()))
        row["mode"] = "walk" if B >= sdva.LAZY_WALK_MIN_LANES else "parallel"
        row["max_accept_len"] = int(acc.max().item())
        row["rows_needed"] = int((acc + 1).sum().item())
        res[str(B)] = row
        del logits
    print(json.dumps({"lazy_sweep": res, "vocab": V, "window": W, "p": p, "steps": args.steps,
                      "warmup": args.warmup}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(all_workload_specs()))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-workloads", action="store_true",
                    help="skip the all_workloads object (every workload's verify_attn and step times)")
    ap.add_argument("--lazy-sweep", action="store_true",
                    help="time spec_accept vs spec_accept_lazy over lane counts instead of the step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.lazy_sweep:
        return run_lazy_sweep(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
