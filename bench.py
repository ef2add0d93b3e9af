#!/usr/bin/env python
"""Benchmark of the verify step (kv_append_quant -> verify_attn -> spec_accept).

Default workload: 8 lanes with contexts uniform in [4096, 65536], 24 q / 4 kv
heads, head_dim 128, window 1 + 15 drafts, FP8 E4M3 KV (page 64, permuted page
table), acceptance over a 151,936-token vocabulary.  Inputs are seeded and
synthetic and already resident in HBM when the timed region starts.

One JSON line (rank 0):
  value        verify steps/s (append + verify_attn + spec_accept), device time
  verify_attn  achieved algorithmic HBM GB/s of the verify_attn call and its
               fraction of the measured copy bandwidth (roofline object)
  e2e          the same steps/s through the C ABI from pinned HOST buffers,
               host->device inputs and device->host results inside the timing
               (the logits copy overlaps append and verify: only accept reads it)
  cpu_baseline the CPU oracle on the host cores, on a bounded sample
  spec_accept_lazy  the acceptance that reads each lane's logits rows only up
               to its first disagreement (timed apart, after the main loop),
               with the step rate it would give
  spec_accept_sampled  lossless stochastic acceptance with a synthetic draft
               distribution (timed apart likewise)
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
# measured by ncu for the current kernels, per workload (absent: not captured
# for this workload, reported as null).  Source: the ncu launch-list summary
# of the multi-lane workload under profiles/.
NCU_TRAFFIC_BYTES = {"multi_lane": 305_100_032 + 742_400 + 8_818_432}


def workload_desc(spec: synth.Spec) -> str:
    kv = "FP8 E4M3 KV, fp32 scale per (page, head)" if spec.kv_dtype == synth.KV_FP8 else \
        "INT4 KV, fp16 scale per group of 32"
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
        kv = tokens * Hkv * 256 + pages * Hkv * 8
    else:
        kv = tokens * Hkv * (128 + 16)
    qo = 2 * len(seq_lens) * W * Hq * 128 * 2
    return kv + qo + pages * 4 + len(seq_lens) * 4


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


def oracle_sample_step(spec, step, cache, rows, threads):
    """One bounded sample of a step on the CPU oracle, scaled to a full step.
    Returns (estimated full-step seconds, sample seconds)."""
    import oracle
    B, W, Hq = step.q.shape[:3]
    sample_lanes = sorted({r[0] for r in rows})
    c = cache.copy()
    t0 = time.perf_counter()
    sel = np.array(sample_lanes)
    oracle.append(c, step.k_win[sel], step.v_win[sel], step.page_table[sel], step.seq_lens[sel])
    t_app = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.verify_attn(c, step.q, step.page_table, step.seq_lens, SM_SCALE, rows=rows, threads=threads)
    t_att = time.perf_counter() - t0
    t_acc = 0.0
    if step.logits is not None:
        t0 = time.perf_counter()
        oracle.spec_accept(step.logits[sel[:1]], step.drafts[sel[:1]], step.seq_lens[sel[:1]])
        t_acc = (time.perf_counter() - t0) * B
    # attention work is proportional to visible keys per row
    full = sum(W * Hq * (int(L) + (W + 1) / 2) for L in step.seq_lens)
    part = sum(int(step.seq_lens[b]) + i + 1 for (b, i, h) in rows)
    est = t_app * B / len(sample_lanes) + t_att * full / part + t_acc
    return est, t_app + t_att + t_acc / B


def sample_rows(step, lanes, n, seed):
    rng = np.random.default_rng(seed)
    B, W, Hq = step.q.shape[:3]
    return [(int(rng.choice(lanes)), int(rng.integers(0, W)), int(rng.integers(0, Hq))) for _ in range(n)]


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    spec = synth.WORKLOADS[args.workload]
    step = synth.make_step(spec)
    lanes = [0, 1] if spec.num_lanes > 1 else [0]
    cache = oracle_setup(spec, step, lanes)
    threads = os.cpu_count() or 1
    ests = []
    for k in range(args.warmup + args.steps):
        rows = sample_rows(step, lanes, threads, 1000 + k)
        est, _ = oracle_sample_step(spec, step, cache, rows, threads)
        if k >= args.warmup:
            ests.append(est)
    sec = float(np.mean(ests))
    value = 1.0 / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": workload_desc(spec)},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: window append of {len(lanes)} lanes, {threads} attention rows "
                                   f"(fp64, {threads} threads), acceptance of 1 lane; scaled to the full step by "
                                   f"visible-key count and lane count"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import speculative_decode_verify_append_gb300 as sdva
    from speculative_decode_verify_append_gb300.step import VerifyStep, fill_context

    spec = synth.WORKLOADS[args.workload]
    step = synth.make_step(spec)
    B, W, Hq = step.q.shape[:3]
    Hkv = spec.num_kv_heads
    max_context = spec.ctx_hi

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    # ---- resident state: cache filled by the library's own append ----
    cache = sdva.KVCache(spec.kv_dtype, step.num_pages, Hkv, device=dev)
    table = torch.from_numpy(step.page_table).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for b in range(B):
        L = int(step.seq_lens[b])
        for start, n in synth.fill_chunks(L, 16384):
            k, v = synth.context_chunk(spec, b, start, n)
            fill_context(cache, bf16(k), bf16(v), table[b], start=start, chunk=4096, status=status)
    torch.cuda.synchronize()
    seq = torch.from_numpy(step.seq_lens).to(dev)
    commit_lens = seq.clone()  # the commit advances a copy: the timed steps keep the same work
    q, kw, vw = bf16(step.q), bf16(step.k_win), bf16(step.v_win)
    logits = torch.from_numpy(step.logits).to(dev) if step.logits is not None else None
    drafts = torch.from_numpy(step.drafts).to(dev) if step.drafts is not None else None
    vs = VerifyStep(B, W, Hq, Hkv, max_context, spec.vocab, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        # The write evicts the step's inputs; the read of a second buffer then
        # evicts the write's dirty lines, whose write-back would otherwise land
        # inside the timed step.
        flush.zero_()
        clean.amax()
    stream = torch.cuda.current_stream()

    def one_step(evs=None):
        if evs:
            evs[0].record(stream)
        vs.append(cache, kw, vw, table, seq)
        if evs:
            evs[1].record(stream)
        vs.attend(cache, q, table, seq)
        if evs:
            evs[2].record(stream)
        if logits is not None:
            vs.accept(logits, drafts, commit_lens)
        if evs:
            evs[3].record(stream)

    for _ in range(args.warmup):
        flush_l2()
        one_step()
    torch.cuda.synchronize()
    assert int(vs.status.item()) == 0, sdva.sdva_status_string(int(vs.status.item()))

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler see the GPU under load from the first step
    wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed_steps")
    for k in range(args.steps):
        flush_l2()
        one_step(evs[k])
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(dist)
    clocks = sampler.stop()
    t_app = [e[0].elapsed_time(e[1]) for e in evs]
    t_att = [e[1].elapsed_time(e[2]) for e in evs]
    t_acc = [e[2].elapsed_time(e[3]) for e in evs]
    t_step = [e[0].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(dist, float(np.sum(t_step)))
    ms_per_step = total_ms / args.steps
    value = world * args.steps / (total_ms / 1e3)

    # ---- lazy acceptance (rows read only up to each lane's first disagreement) ----
    lazy = None
    if logits is not None:
        l_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.warmup + args.steps):
            flush_l2()
            if k >= args.warmup:
                l_ev[k - args.warmup][0].record(stream)
            vs.accept_lazy(logits, drafts, None, commit_lens)
            if k >= args.warmup:
                l_ev[k - args.warmup][1].record(stream)
        torch.cuda.synchronize()
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
        s_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.warmup + args.steps):
            flush_l2()
            if k >= args.warmup:
                s_ev[k - args.warmup][0].record(stream)
            sdva.spec_accept_sampled(logits, qd, dq, ua, us, s_acc, s_tok, ws, commit_lens, vs.status)
            if k >= args.warmup:
                s_ev[k - args.warmup][1].record(stream)
        torch.cuda.synchronize()
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

    # ---- e2e: host buffers through the public API ----
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
    # their copy runs in two halves on two side streams, beside append and
    # verify, and accept waits for it.  Each step's copies start inside its
    # timed region (the side streams wait for everything issued before it).
    side = [torch.cuda.Stream(device=dev) for _ in range(2)]
    for k in range(e2e_steps + 3):
        flush_l2()
        if k >= 3:
            e_ev[k - 3][0].record(stream)
        logits_ready = []
        if logits is not None:
            half = logits.shape[0] // 2 if logits.shape[0] > 1 else logits.shape[0]
            parts = [(0, half), (half, logits.shape[0])] if half < logits.shape[0] else [(0, logits.shape[0])]
            for (lo, hi), cs in zip(parts, side):
                cs.wait_stream(stream)  # the previous step's accept has read the old logits
                with torch.cuda.stream(cs):
                    dev_in["logits"][lo:hi].copy_(host_in["logits"][lo:hi], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                logits_ready.append(ev)
        for n, t in host_in.items():
            if n != "logits":
                dev_in[n].copy_(t, non_blocking=True)
        vs.append(cache, kw, vw, table, seq)
        vs.attend(cache, q, table, seq)
        if logits is not None:
            for ev in logits_ready:
                stream.wait_event(ev)
            vs.accept(logits, drafts, commit_lens)
        host_out["out"].copy_(vs.out, non_blocking=True)
        if logits is not None:
            host_out["acc"].copy_(vs.accept_len, non_blocking=True)
            host_out["tok"].copy_(vs.out_tokens, non_blocking=True)
        if k >= 3:
            e_ev[k - 3][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, float(np.sum([e[0].elapsed_time(e[1]) for e in e_ev])))
    e2e_value = world * e2e_steps / (e2e_ms / 1e3)

    # ---- roofline of the verify_attn call ----
    alg = verify_algorithmic_bytes(spec, step.seq_lens)
    att_ms = float(np.mean(t_att))
    achieved = alg / (att_ms / 1e3) / 1e9
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"]
    traffic = NCU_TRAFFIC_BYTES.get(spec.name)

    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8-e4m3 KV (int4 for the 4-bit workload) -> f16 tensor-core MMA, f32 accumulate, bf16 out",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, N(0,1) fp32 logits)",
        "config": {"workload": workload_desc(spec), "lanes": B, "window": W, "q_heads": Hq, "kv_heads": Hkv,
                   "context_tokens": int(step.seq_lens.sum()), "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed step (512 MB write, then 512 MB read of a second buffer; untimed)"},
        "verify_attn": {"us": att_ms * 1e3, "gbs": achieved, "pct_of_peak": 100.0 * achieved / peak,
                        "algorithmic_bytes": alg},
        "breakdown_us": {"kv_append_quant": float(np.mean(t_app)) * 1e3, "verify_attn": att_ms * 1e3,
                         "spec_accept": float(np.mean(t_acc)) * 1e3},
        "roofline": {"kernel": "verify_attn (split-K + merge kernels)", "bound": "hbm", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic, "algorithmic_bytes": alg},
        "e2e": {"value": e2e_value, "unit": "steps/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "spec_accept_lazy": lazy,
        "spec_accept_sampled": sampled,
        "gpu_launches": args.steps * (1 + 2 + (2 if logits is not None else 0)),
        "clocks": clocks,
        "wall_s_timed_loop": wall,
    }

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        lanes = [0, 1] if B > 1 else [0]
        ocache = oracle_setup(spec, step, lanes)
        threads = os.cpu_count() or 1
        ests = []
        t_budget = time.perf_counter()
        k = 0
        while (k < 3 or time.perf_counter() - t_budget < 10.0) and k < 20:
            rows = sample_rows(step, lanes, threads, 77 + k)
            est, _ = oracle_sample_step(spec, step, ocache, rows, threads)
            ests.append(est)
            k += 1
        line["cpu_baseline"] = {
            "value": 1.0 / float(np.mean(ests)), "unit": "steps/s", "cores": threads, "kind": "oracle",
            "sample": f"{k} samples of: window append of {len(lanes)} lanes, {threads} random attention rows "
                      f"(fp64, {threads} threads), acceptance of 1 lane; scaled to a full step by visible keys "
                      f"and lanes"}
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
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
