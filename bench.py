#!/usr/bin/env python3
"""Benchmark of paged FP8 attention on GB300.

One step = one pass of the whole hot path over one batch: Q -> E4M3 (FP8-MMA
workloads), the device-side plan, the attention kernel(s) and the split-KV
combine, through the library's C ABI.  Inputs are resident in HBM when the
timed region starts.  Decode, verify and mixed batches are measured in
KV-cache bytes read per second (algorithmic bytes: the K and V rows of every
(sequence, KV head) visible key range, counted once), the decode roofline;
the 4096-token chunk alone (chunk_* workloads) in TFLOP/s of visible QK^T and
PV work against the dense tensor peak.  The kv_write_* workloads time the
paged KV-cache write instead (bf16 K/V read plus E4M3 bytes written, per
second), lse_combine_* the merge of DCP partials.

The default workload is the largest one that fits one GPU: the chunked-prefill
mixed batch at head dim 512 (4096-token chunk on 4096 cached keys plus 4032
decode sequences, BF16 Q, 71.9 GB of K/V read per step).  A one-GPU run then
also measures every other attention workload and reports each in the line's
per_config block (kernel time, roofline fraction, clocks).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (the attention op has no exchange
step), the timed region is bracketed by barriers and the slowest rank's time
is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

DEFAULT_CONFIG = "mixed_hd512_causal"
METRIC = "paged FP8 attn: prefill TFLOP/s & decode KV GB/s, % of GB300 roofline"
KERNEL_SOURCES = ["attn_kernel.cuh", "attn_prefill.cuh", "common.cuh", "ptx.cuh", "attn_launch.cuh"]
KV_WRITE_SOURCES = ["kv_cache_write.cu", "quant_e4m3.cuh"]
COMBINE_SOURCES = ["lse_combine.cu"]


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]), source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, "fp8_paged_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(config: str, sources=None):
    """DRAM bytes per launch of the workload's main kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(config)
        if e and e.get("kernel_source_sha") == kernel_source_hash(sources):
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region.  Samples
    carry nvidia-smi's own timestamp; mark() brackets the timed region on the
    host clock, and the summary keeps only the samples inside it (all samples
    when the region was too short to hold one)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 25

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, t0: float, t1: float):
        """Host wall-clock times (time.time()) of the timed region's start and end."""
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        sm, smax = float(parts[2]), float(parts[3])
                    except ValueError:
                        continue
                    act = {n for n, v in zip(names, parts[6:10]) if v.lower() == "active"}
                    rows.append((ts, sm, smax, act))
            os.unlink(self.path)
        except Exception:
            return None
        if not rows:
            return None
        window = "timed region"
        if self.t0 is not None:
            inside = [r for r in rows if self.t0 <= r[0] <= self.t1]
            if inside:
                rows_used = inside
            else:
                rows_used, window = rows, "whole sampler run (timed region shorter than the sampling period)"
        else:
            rows_used, window = rows, "whole sampler run"
        reasons = set().union(*[r[3] for r in rows_used])
        return {"sm_mhz": statistics.median(r[1] for r in rows_used), "sm_max_mhz": max(r[2] for r in rows_used),
                "reasons": sorted(reasons), "samples": len(rows_used), "period_ms": self.PERIOD_MS,
                "window": window}


def unit_bytes_of(w: synth.Workload, units):
    """Algorithmic K+V bytes of a set of (sequence, kv-head) units."""
    total = 0
    for b, _hk in units:
        span = synth._seq_visible_span(int(w.lq[b]), int(w.lk[b]), w.window_left, w.causal)
        if span is not None:
            total += (span[1] - span[0] + 1) * w.head_dim * 2
    return total


# ------------------------------------------------------------------ CPU oracle leg

def unit_flops_of(w: synth.Workload, units):
    """QK^T + PV flops (4 D per visible pair) of a set of (sequence, kv-head) units."""
    G = w.num_heads_q // w.num_heads_kv
    return sum(synth._visible_count(int(w.lq[b]), int(w.lk[b]), w.window_left, w.causal) * G * 4 * w.head_dim
               for b, _hk in units)


def oracle_timing(w: synth.Workload, budget_s: float, seed: int = 0, tflops: bool = False):
    """Time the oracle on a bounded sample of (sequence, kv-head) units of the
    workload (every query row and head of each unit).  Returns (rate in GB/s,
    or TFLOP/s when tflops, cores, description, seconds)."""
    import oracle  # test/benchmark infrastructure only
    rng = np.random.default_rng(seed)
    G = w.num_heads_q // w.num_heads_kv
    units_all = [(b, hk) for b in range(w.batch) if w.lq[b] > 0 for hk in range(w.num_heads_kv)]
    order = rng.permutation(len(units_all))
    cu = np.zeros(w.batch + 1, dtype=np.int64)
    cu[1:] = np.cumsum(w.lq)

    def run(units):
        seqs = sorted({b for b, _ in units})
        sub = synth.subproblem_pages(w, seqs)
        q = sub["q"]
        if w.fp8_q:
            q = oracle.quantize_q(q, w.q_descale)
        prob = oracle.AttnProblem(q, w.fp8_q, sub["k"], sub["v"], sub["block_table"], sub["cu_seqlens_q"],
                                  sub["seqused_k"], w.num_heads_kv, w.q_descale, w.k_descale, w.v_descale,
                                  w.softmax_scale, w.window_left, w.causal)
        local = {b: i for i, b in enumerate(seqs)}
        rows = []
        for b, hk in units:
            i = local[b]
            for t in range(sub["cu_seqlens_q"][i], sub["cu_seqlens_q"][i + 1]):
                for g in range(G):
                    rows.append((t, hk * G + g))
        rows = np.array(rows, dtype=np.int32)
        t0 = time.perf_counter()
        oracle.paged_attention(prob, rows=rows)
        return time.perf_counter() - t0

    # pilot on a few units, then size the sample to the budget
    n = min(len(units_all), 8)
    pilot = [units_all[i] for i in order[:n]]
    t = run(pilot)
    pilot_rate = unit_flops_of(w, pilot) / max(t, 1e-9)
    want = budget_s * pilot_rate
    units, acc = [], 0
    for i in order:
        units.append(units_all[i])
        acc += unit_flops_of(w, [units_all[i]])
        if acc >= want:
            break
    t = run(units)
    rate = unit_flops_of(w, units) / t / 1e12 if tflops else unit_bytes_of(w, units) / t / 1e9
    cores = os.cpu_count() or 1
    desc = (f"{len(units)} of {len(units_all)} (sequence, KV head) units of {w.name}, every query row and head; "
            f"{unit_bytes_of(w, units) / 1e6:.1f} MB of algorithmic KV bytes, "
            f"{unit_flops_of(w, units) / 1e9:.2f} GFLOP, in {t:.2f} s")
    return rate, cores, desc, t


def kv_write_oracle_timing(w, budget_s: float, seed: int = 0):
    """Time the oracle's KV-cache write on a bounded sample of the workload's
    tokens.  Returns (GB/s of algorithmic bytes, cores, description, seconds)."""
    import oracle  # test/benchmark infrastructure only
    rng = np.random.default_rng(seed)
    kb = w.key.cpu().view(torch.int16).numpy().view(np.uint16)
    vb = w.value.cpu().view(torch.int16).numpy().view(np.uint16)
    sm = w.slot_mappings[0].cpu().numpy()
    per_token = w.num_heads_kv * w.head_dim * 2 * 3
    order = rng.permutation(w.num_tokens)

    def run(idx):
        pages = np.unique(sm[idx] // synth.PAGE)
        local = {int(p): i for i, p in enumerate(pages)}
        slots = np.array([local[int(x) // synth.PAGE] * synth.PAGE + int(x) % synth.PAGE for x in sm[idx]], np.int64)
        kc = np.zeros((len(pages), synth.PAGE, w.num_heads_kv, w.head_dim), np.uint8)
        vc = np.zeros_like(kc)
        k, v = np.ascontiguousarray(kb[idx]), np.ascontiguousarray(vb[idx])
        t0 = time.perf_counter()
        oracle.kv_cache_write(k, v, slots, w.k_descale, w.v_descale, kc, vc)
        return time.perf_counter() - t0

    pilot = order[:64]
    t = run(pilot)
    n = int(min(w.num_tokens, max(64, budget_s / max(t, 1e-9) * len(pilot))))
    idx = order[:n]
    t = run(idx)
    desc = (f"{n} of {w.num_tokens} tokens of {w.name} ({n * per_token / 1e6:.1f} MB of algorithmic bytes) "
            f"in {t:.2f} s, one thread")
    return n * per_token / t / 1e9, 1, desc, t


def combine_oracle_timing(w, budget_s: float):
    """Time the oracle's LSE combine on a bounded sample of rows (tokens)."""
    import oracle  # test/benchmark infrastructure only
    P, T, hq, d = w.o_parts.shape
    ob = w.o_parts.cpu().view(torch.int16).numpy().view(np.uint16)
    lb = w.lse_parts.cpu().numpy()
    per_tok = (P + 1) * hq * (2 * d + 4)

    def run(n):
        o = np.ascontiguousarray(ob[:, :n])
        ls = np.ascontiguousarray(lb[:, :, :n])
        t0 = time.perf_counter()
        oracle.lse_combine(o, ls)
        return time.perf_counter() - t0

    t = run(16)
    n = int(min(T, max(16, budget_s / max(t, 1e-9) * 16)))
    t = run(n)
    desc = f"{n} of {T} tokens of {w.name} ({n * per_tok / 1e6:.1f} MB of algorithmic bytes) in {t:.2f} s, one thread"
    return n * per_tok / t / 1e9, 1, desc, t


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    if args.config in synth.COMBINE_CONFIG_NAMES:
        w = synth.make_combine_config(args.config)
        total_steps = args.steps + args.warmup
        per_step = max(0.05, min(30.0, 150.0 / max(1, total_steps)))
        vals, t_all, desc, cores = [], 0.0, "", 1
        for i in range(total_steps):
            r, cores, desc, t = combine_oracle_timing(w, per_step)
            if i >= args.warmup:
                vals.append(r)
                t_all += t
        value = statistics.median(vals)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_all / max(1, len(vals)), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": "per step: " + desc},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0
    if args.config in synth.KV_WRITE_CONFIG_NAMES:
        w = synth.make_kv_write_config(args.config)
        total_steps = args.steps + args.warmup
        per_step = max(0.05, min(30.0, 150.0 / max(1, total_steps)))
        vals, t_all, desc, cores = [], 0.0, "", 1
        for i in range(total_steps):
            r, cores, desc, t = kv_write_oracle_timing(w, per_step, seed=i)
            if i >= args.warmup:
                vals.append(r)
                t_all += t
        value = statistics.median(vals)
        line = {
            "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_all / max(1, len(vals)), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 -> e4m3",
            "data": "synthetic", "config": {"workload": w.name, "sample": "per step: " + desc},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return 0
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.make_config(args.config, device=dev)
    total_steps = args.steps + args.warmup
    per_step = max(0.05, min(30.0, 150.0 / max(1, total_steps)))
    vals, cores, desc = [], 1, ""
    t_all = 0.0
    tensor_bound = w.name.startswith("chunk_")
    unit = "TFLOP/s" if tensor_bound else "GB/s"
    for i in range(total_steps):
        r, cores, desc, t = oracle_timing(w, per_step, seed=i, tflops=tensor_bound)
        if i >= args.warmup:
            vals.append(r)
            t_all += t
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * t_all / max(1, len(vals)), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": "per step: " + desc},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ replicas across ranks

def hold_device(steps: int, host_us_per_step: float = 100.0, margin_us: float = 100000.0):
    """Enqueues a device-side wait of at least `steps * host_us_per_step +
    margin_us` us on the current stream just before a timed region.  The host
    then queues every timed launch while the GPU waits, so a kernel shorter than
    its own host-side submission does not sit idle inside its timed interval
    waiting for the launch to arrive; the margin absorbs a stall of the host
    thread while it queues (one such stall of ~80 ms once stretched a 10 ms
    region ninefold).  Torch's spin kernel, clock cycles at the highest SM
    clock; it runs before the region's first event and is not part of any
    timing."""
    us = min(steps * host_us_per_step + margin_us, 600000.0)
    torch.cuda._sleep(int(us * 2070))


def time_single_launch(step, first: int, steps: int, stream, world: int, dev, local_rank: int):
    """Times a step that is exactly one launch of one kernel.  Region: `steps`
    launches back to back between two events (nothing else inside), with clocks
    sampled; its mean is the launch duration the roofline uses.  Then `steps`
    more launches, each between its own pair of events: that mean also holds the
    events' own cost (a few microseconds per launch, which weighs on a kernel of
    tens of microseconds) and is reported beside it.  step(i) runs launch i.
    Returns (region ms over all steps, max over ranks; region mean ms per launch;
    per-launch event mean ms; clock record)."""
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    h0 = time.time()
    hold_device(steps)
    t_start.record(stream)
    for i in range(steps):
        step(first + i)
    t_stop.record(stream)
    torch.cuda.synchronize()
    clocks.mark(h0, time.time())
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop()
    ms_total = slowest_rank_ms(t_start.elapsed_time(t_stop), world, dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    hold_device(steps)
    for i in range(steps):
        ev[i][0].record(stream)
        step(first + steps + i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ev_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    return ms_total, ms_total / steps, ev_ms, clock_info


def slowest_rank_ms(ms: float, world: int, device) -> float:
    """The whole job's time of a replicated (weak-scaling) run: the maximum over
    ranks of each rank's elapsed milliseconds."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_step: float, world: int, steps: int, ms_total: float, tflops: bool) -> float:
    """Whole-job throughput: the work of every rank's steps over the slowest rank's time."""
    return world * work_per_step * steps / (ms_total * 1e-3) / (1e12 if tflops else 1e9)


# ------------------------------------------------------------------ GPU leg

def unique_kv_bytes(w: synth.Workload) -> int:
    """K+V bytes of the distinct physical pages that visible keys sit in,
    counting each page's visible slots once however many sequences share it
    (the speculative-verify batch's prefix pages are shared by every sequence)."""
    slots = {}
    for b in range(w.batch):
        span = synth._seq_visible_span(int(w.lq[b]), int(w.lk[b]), w.window_left, w.causal)
        if span is None:
            continue
        lo, hi = span
        for j in range(lo // synth.PAGE, hi // synth.PAGE + 1):
            a, e = max(lo, j * synth.PAGE), min(hi, j * synth.PAGE + synth.PAGE - 1)
            phys = int(w.bt[b, j])
            slots[phys] = max(slots.get(phys, 0), e - a + 1)
    return sum(slots.values()) * w.num_heads_kv * w.head_dim * 2


# The workloads the default run measures after its headline line, each in one
# entry of the line's per_config block: the decode and verify configurations,
# the other mixed batches, the 4096-token chunk alone (prefill, tensor-bound)
# and the tiny prefill.
PER_CONFIG = ["swa_decode_hd256", "full_decode_hd512_bf16q", "full_decode_hd512_fp8q", "spec_verify_hd512",
              "mixed_hd256_swa", "mixed_hd512_causal", "mixed_hd512_causal_fp8q", "chunk_hd256_swa",
              "chunk_hd512_causal", "chunk_hd512_causal_fp8q", "tiny_prefill_hd256"]


def time_workload(w: synth.Workload, args, dev, world: int, steps: int, warmup: int, with_e2e: bool):
    """Times `steps` forward steps of one workload (after `warmup` untimed
    ones) with inputs resident, the attention kernels alone on CUDA events, and
    optionally the end-to-end loop through the public call with host buffers.
    Returns a dict of the measurements."""
    import fp8_paged_attention_gb300 as fp8pa  # the CUDA library; raises if it cannot load
    stream = torch.cuda.current_stream()
    qd = torch.tensor([w.q_descale], dtype=torch.float32, device=dev)
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device=dev)
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device=dev)
    hq, hkv, D = w.num_heads_q, w.num_heads_kv, w.head_dim
    max_pages = w.block_table.shape[1]
    qdt = fp8pa.FP8PA_E4M3 if w.fp8_q else fp8pa.FP8PA_BF16
    ns_arg = args.num_splits
    ws_bytes = fp8pa.workspace_size(w.batch, w.total_q, w.max_seqlen_q, hq, hkv, D, qdt, max_pages, w.window_left,
                                    ns_arg)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((w.total_q, hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((hq, w.total_q), dtype=torch.float32, device=dev)
    q8 = torch.empty((w.total_q, hq, D), dtype=torch.uint8, device=dev)
    splits = fp8pa.num_splits(w.batch, w.total_q, w.max_seqlen_q, hq, hkv, D, qdt, max_pages, w.window_left, ns_arg)
    launches = fp8pa.kernel_launches(w.batch, w.total_q, w.max_seqlen_q, hq, hkv, D, qdt, max_pages, w.window_left,
                                     ns_arg)
    launches += 1 if w.fp8_q else 0

    # A step must not find its inputs in L2 from the step before.  Where one
    # step's working set (K/V cache, Q, out, lse) is smaller than three times
    # the L2, the steps rotate over enough independent copies of it.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = sum(t.numel() * t.element_size() for t in (w.k_cache, w.v_cache, w.q, out, lse))
    n_rot = 1 if per_copy >= 3 * l2_bytes else min(1024, -(-3 * l2_bytes // per_copy))
    kv_rot = [(w.k_cache, w.v_cache)] + [(w.k_cache.clone(), w.v_cache.clone()) for _ in range(n_rot - 1)]
    q_rot = [w.q] + [w.q.clone() for _ in range(n_rot - 1)]
    ol_rot = [(out, lse)] + [(torch.empty_like(out), torch.empty_like(lse)) for _ in range(n_rot - 1)]
    if n_rot > 1:
        l2_note = (f"inputs rotated over {n_rot} copies of {per_copy / 1e6:.1f} MB "
                   f"({n_rot * per_copy / 1e6:.0f} MB, over 3x the {l2_bytes / 1e6:.0f} MB L2)")
    else:
        l2_note = (f"inputs larger than L2: {per_copy / 1e6:.0f} MB of cache, Q and outputs, "
                   f"{w.kv_bytes_algorithmic() / 1e6:.0f} MB of K/V read per step, {l2_bytes / 1e6:.0f} MB L2")

    # attention sinks (one logit per query head), drawn N(0, 1), when asked for
    sinks = (torch.randn(hq, generator=torch.Generator().manual_seed(3)).to(dev) if args.sinks else None)

    def step(q_src, bt, cu, su, o, l, r=0):
        kc, vc = kv_rot[r % n_rot]
        q = fp8pa.quantize_q_fp8(q_src, qd, out=q8) if w.fp8_q else q_src
        fp8pa.fp8_paged_attn_fwd(q, kc, vc, bt, cu, su, w.max_seqlen_q, qd, kd, vd,
                                 w.softmax_scale, w.window_left, w.causal, num_splits=ns_arg, out=o, lse=l,
                                 workspace=workspace, sinks=sinks)

    def args_dev(i):
        o, l = ol_rot[i % n_rot]
        return (q_rot[i % n_rot], w.block_table, w.cu_seqlens_q, w.seqused_k, o, l, i)

    for i in range(warmup):
        step(*args_dev(i))
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---------------- device-resident timed region: `steps` steps back to back, nothing
    # between their launches (an event recorded between the plan and the attention kernel
    # would break their programmatic overlap and slow the step)
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    h0 = time.time()
    hold_device(steps)
    t_start.record(stream)
    for i in range(steps):
        step(*args_dev(warmup + i))
    t_stop.record(stream)
    torch.cuda.synchronize()
    clocks.mark(h0, time.time())
    barrier()
    clock_info = clocks.stop()
    ms_total = t_start.elapsed_time(t_stop)
    # ---------------- the attention kernels alone: `steps` more steps, each with CUDA events
    # recorded on the launching stream just before the first attention kernel and just after
    # the last (fp8pa_set_timing_events)
    k_start = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    k_stop = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in k_start + k_stop:
        e.record(stream)  # torch creates the CUDA event on first record; the library re-records it
    torch.cuda.synchronize()
    hold_device(steps)
    for i in range(steps):
        fp8pa.set_timing_events(k_start[i], k_stop[i])
        step(*args_dev(warmup + steps + i))
    fp8pa.set_timing_events(None, None)
    torch.cuda.synchronize()
    k_ms = [a.elapsed_time(b) for a, b in zip(k_start, k_stop)]
    ms_total = slowest_rank_ms(ms_total, world, dev)
    kv_bytes = w.kv_bytes_algorithmic()
    peaks = measured_peaks()
    k_avg_ms = sum(k_ms) / len(k_ms)
    tensor_bound = w.name.startswith("chunk_")
    # prefill-class row tiles with E4M3 Q run the rows-on-lanes prefill kernel, all others attn_fwd_kernel
    prefill_tiles = w.max_seqlen_q * (hq // hkv) > 32
    if w.fp8_q and prefill_tiles:
        kernel = "attn_prefill_kernel" if w.name.startswith("chunk_") else \
            "attn_fwd_kernel (decode rows) + attn_prefill_kernel (chunk rows)"
    else:
        kernel = "attn_fwd_kernel"
    if tensor_bound:
        # a prefill chunk alone: causal/window-visible QK^T + PV flops against the dense tensor peak
        flops = w.flops_algorithmic()
        unit = "TFLOP/s"
        value = job_rate(flops, world, steps, ms_total, True)
        achieved = flops / (k_avg_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"] * (2.0 if w.fp8_q else 1.0)
        peak_src = (peaks["source"] + " MEASURED_PEAKS.json bf16_tflops (burst)" +
                    (" x 2, the nominal FP8/BF16 dense ratio" if w.fp8_q else ""))
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": unit,
                    "frac": round(achieved / peak, 4), "traffic": ncu_traffic(w.name),
                    "kernel": kernel, "kernel_ms": round(k_avg_ms, 5), "peak_source": peak_src}
    else:
        unit = "GB/s"
        value = job_rate(kv_bytes, world, steps, ms_total, False)
        achieved = kv_bytes / (k_avg_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": unit,
                    "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": ncu_traffic(w.name),
                    "kernel": kernel, "kernel_ms": round(k_avg_ms, 5),
                    "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"}
        ub = unique_kv_bytes(w)
        if ub < kv_bytes:
            # pages shared by several sequences: their bytes can come from L2 after the first read
            roofline["unique_bytes"] = ub
            roofline["unique_achieved"] = round(ub / (k_avg_ms * 1e-3) / 1e9, 2)
            roofline["unique_frac"] = round(ub / (k_avg_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)

    def rate(n_steps, ms):
        work = w.flops_algorithmic() if tensor_bound else kv_bytes
        return job_rate(work, world, n_steps, ms, tensor_bound)

    # ---------------- end to end through the public API, host buffers
    # Every step copies its inputs (Q, block table, lengths) from pinned host memory
    # and reads its result (out, lse) back.  As in a serving loop, uploads and
    # read-backs run on streams of their own, overlapping the compute of the
    # neighbouring steps: two device buffer sets, ordered by events.  The timed
    # region runs from the first upload to the end of the last read-back.
    e2e = None
    if with_e2e:
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        h_q, h_bt, h_cu, h_su = pin(w.q), pin(w.block_table), pin(w.cu_seqlens_q), pin(w.seqused_k)
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        sets = []
        for _ in range(2):
            sets.append(dict(q=torch.empty_like(w.q), bt=torch.empty_like(w.block_table),
                             cu=torch.empty_like(w.cu_seqlens_q), su=torch.empty_like(w.seqused_k),
                             out=torch.empty_like(out), lse=torch.empty_like(lse),
                             up=torch.cuda.Event(), done=torch.cuda.Event(), back=torch.cuda.Event()))
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_bt, h_cu, h_su))
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
        up_stream, down_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_run(n, first):
            for i in range(n):
                b = sets[i & 1]
                with torch.cuda.stream(up_stream):
                    if not (first and i < 2):
                        up_stream.wait_event(b["done"])  # step i - 2 has read this set's inputs
                    b["q"].copy_(h_q, non_blocking=True)
                    b["bt"].copy_(h_bt, non_blocking=True)
                    b["cu"].copy_(h_cu, non_blocking=True)
                    b["su"].copy_(h_su, non_blocking=True)
                    b["up"].record(up_stream)
                stream.wait_event(b["up"])
                if not (first and i < 2):
                    stream.wait_event(b["back"])  # step i - 2's result has left this set's outputs
                step(b["q"], b["bt"], b["cu"], b["su"], b["out"], b["lse"], i)
                b["done"].record(stream)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(b["done"])
                    h_out.copy_(b["out"], non_blocking=True)
                    h_lse.copy_(b["lse"], non_blocking=True)
                    b["back"].record(down_stream)

        e2e_run(max(3, warmup // 4), True)
        torch.cuda.synchronize()
        # the first upload and the last read-back lie outside the overlap: enough
        # steps that they weigh little against the steady state a serving loop runs in
        n_e2e = max(40, steps // 2)
        barrier()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(up_stream)
        e2e_run(n_e2e, False)
        e.record(down_stream)
        torch.cuda.synchronize()
        e_ms = a.elapsed_time(e)
        e_ms = slowest_rank_ms(e_ms, world, dev)
        e2e = {"value": round(rate(n_e2e, e_ms), 3), "unit": unit,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "ms_per_step": round(e_ms / n_e2e, 5),
               "note": "K/V cache is resident state; per step Q, block table and lengths go up and out and lse "
                       "come back, on copy streams overlapping the neighbouring steps' compute"}
    roofline["kernel_timing"] = ("CUDA events around the attention kernels on the launching stream, over a "
                                 "second pass of the same number of steps right after the timed region")
    return dict(value=value, unit=unit, ms_per_step=ms_total / steps, roofline=roofline, e2e=e2e, clocks=clock_info,
                splits=splits, launches=launches, l2_note=l2_note, kv_bytes=kv_bytes, tensor_bound=tensor_bound)


def config_of(w: synth.Workload, r: dict, world: int, sinks: bool) -> dict:
    return {"workload": w.name, "batch": w.batch, "total_q": w.total_q, "num_heads_q": w.num_heads_q,
            "num_heads_kv": w.num_heads_kv, "head_dim": w.head_dim, "window_left": w.window_left,
            "causal": w.causal, "q": "e4m3" if w.fp8_q else "bf16", "kv": "e4m3, 64-token pages",
            "num_splits": r["splits"], "kv_bytes_per_step": r["kv_bytes"],
            "flops_per_step": w.flops_algorithmic() if r["tensor_bound"] else None,
            "parallelism": f"replicas x{world}", "l2": r["l2_note"], "sinks": bool(sinks)}


def run_ours(args):
    import gc

    rank, local_rank, world = dist_env()
    import fp8_paged_attention_gb300 as fp8pa  # the CUDA library; raises if it cannot load
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    fp8pa.set_ctas_per_sm(args.ctas_per_sm)
    w = synth.make_config(args.config, device=dev)
    r = time_workload(w, args, dev, world, args.steps, args.warmup, with_e2e=not args.no_e2e)
    # ---------------- CPU oracle baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rr, cores, desc, _t = oracle_timing(w, budget_s=args.cpu_budget, tflops=r["tensor_bound"])
        cpu = {"value": round(rr, 6), "unit": r["unit"], "cores": cores, "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": round(r["value"], 3), "unit": r["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if w.fp8_q else "bf16", "data": "synthetic",
        "config": config_of(w, r, world, args.sinks),
        "roofline": r["roofline"], "cpu_baseline": cpu, "e2e": r["e2e"],
        "gpu_launches": r["launches"] * args.steps, "clocks": r["clocks"],
    }
    # ---------------- the other workloads of the metric, one GPU only: kernel and step rates,
    # roofline fraction and clocks of each (no e2e loop, no CPU leg)
    if not args.no_per_config and world == 1:
        del w
        gc.collect()
        torch.cuda.empty_cache()
        per = {}
        steps = args.per_config_steps or args.steps
        for name in PER_CONFIG:
            if name == args.config:
                continue
            wc = synth.make_config(name, device=dev)
            rc = time_workload(wc, args, dev, world, steps, args.warmup, with_e2e=False)
            per[name] = {"value": round(rc["value"], 3), "unit": rc["unit"], "steps": steps,
                         "ms_per_step": round(rc["ms_per_step"], 5), "roofline": rc["roofline"],
                         "clocks": rc["clocks"], "gpu_launches": rc["launches"] * steps,
                         "dtype": "e4m3" if wc.fp8_q else "bf16", "config": config_of(wc, rc, world, args.sinks)}
            del wc
            gc.collect()
            torch.cuda.empty_cache()
        line["per_config"] = per
        line["per_config_note"] = ("each workload timed on its own after the headline's timed region; "
                                   "gpu_launches above counts the headline's timed launches only")
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_kv_write(args):
    """The paged KV-cache write of a mixed batch's new tokens: one launch of
    fp8pa_kv_cache_write per step.  Metric: algorithmic bytes (bf16 K/V read,
    E4M3 written) per second against the HBM copy peak."""
    rank, local_rank, world = dist_env()
    import fp8_paged_attention_gb300 as fp8pa  # the CUDA library; raises if it cannot load
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    probe = synth.make_kv_write_config(args.config)
    per_copy = probe.bytes_algorithmic()
    n_rot = 1 if per_copy >= 3 * l2_bytes else -(-3 * l2_bytes // per_copy)
    w = synth.make_kv_write_config(args.config, device=dev, copies=n_rot)
    keys = [w.key] + [w.key.clone() for _ in range(n_rot - 1)]
    vals = [w.value] + [w.value.clone() for _ in range(n_rot - 1)]
    shape = (w.num_pages, synth.PAGE, w.num_heads_kv, w.head_dim)
    k_cache = torch.empty(shape, dtype=torch.uint8, device=dev)
    v_cache = torch.empty(shape, dtype=torch.uint8, device=dev)
    kd = torch.tensor([w.k_descale], dtype=torch.float32, device=dev)
    vd = torch.tensor([w.v_descale], dtype=torch.float32, device=dev)
    work = w.bytes_algorithmic()

    def step(i, key=None, value=None, slots=None):
        r = i % n_rot
        fp8pa.kv_cache_write(keys[r] if key is None else key, vals[r] if value is None else value, k_cache, v_cache,
                             w.slot_mappings[r] if slots is None else slots, kd, vd)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ms_total, k_avg_ms, k_ev_ms, clock_info = time_single_launch(step, args.warmup, args.steps, stream, world, dev,
                                                                 local_rank)
    value = job_rate(work, world, args.steps, ms_total, False)
    peaks = measured_peaks()
    achieved = work / (k_avg_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": round(peaks["hbm_gbs"], 1), "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": ncu_traffic(w.name, KV_WRITE_SOURCES), "kernel": "kv_cache_write_kernel",
                "kernel_ms": round(k_avg_ms, 5), "kernel_ms_source": "mean over the timed region's back-to-back launches",
                "kernel_ms_events_per_launch": round(k_ev_ms, 5),
                "frac_events_per_launch": round(work / (k_ev_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"] + " MEASURED_PEAKS.json hbm_gbs (copy)"}
    # e2e: each step uploads its keys, values and slot mapping from pinned host
    # memory and reads the device status word back
    e2e = None
    if not args.no_e2e:
        h_k, h_v = w.key.cpu().pin_memory(), w.value.cpu().pin_memory()
        h_s = [m.cpu().pin_memory() for m in w.slot_mappings]
        d_k, d_v = torch.empty_like(w.key), torch.empty_like(w.value)
        d_s = torch.empty_like(w.slot_mappings[0])
        h_status = torch.zeros(1, dtype=torch.int32).pin_memory()
        lib = fp8pa.load_library()

        def e2e_step(i):
            d_k.copy_(h_k, non_blocking=True)
            d_v.copy_(h_v, non_blocking=True)
            d_s.copy_(h_s[i % n_rot], non_blocking=True)
            step(i, d_k, d_v, d_s)
            lib.fp8pa_get_device_status(h_status.data_ptr(), stream.cuda_stream)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(10, args.steps // 4)
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        a.record(stream)
        for i in range(n_e2e):
            e2e_step(i)
        e.record(stream)
        torch.cuda.synchronize()
        e_ms = slowest_rank_ms(a.elapsed_time(e), world, dev)
        h2d = sum(t.numel() * t.element_size() for t in (h_k, h_v, h_s[0]))
        e2e = {"value": round(job_rate(work, world, n_e2e, e_ms, False), 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4, "steps": n_e2e,
               "ms_per_step": round(e_ms / n_e2e, 5),
               "note": "the cache is resident state; per step the keys, values and slot mapping go up and the "
                       "device status word comes back"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, cores, desc, _t = kv_write_oracle_timing(synth.make_kv_write_config(args.config), args.cpu_budget)
        cpu = {"value": round(r, 6), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        l2_note = (f"inputs rotated over {n_rot} copies of {per_copy / 1e6:.1f} MB read and written "
                   f"({n_rot * per_copy / 1e6:.0f} MB, over 3x the {l2_bytes / 1e6:.0f} MB L2)" if n_rot > 1 else
                   f"inputs larger than L2: {per_copy / 1e6:.0f} MB per step")
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_total / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 -> e4m3", "data": "synthetic",
            "config": {"workload": w.name, "num_tokens": w.num_tokens, "num_heads_kv": w.num_heads_kv,
                       "head_dim": w.head_dim, "kv": "e4m3, 64-token pages", "bytes_per_step": work,
                       "parallelism": f"replicas x{world}", "l2": l2_note},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clock_info,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_combine(args):
    """The LSE combine of two DCP shards' partials: one launch of
    fp8pa_lse_combine per step.  Metric: algorithmic bytes per second against
    the HBM copy peak."""
    rank, local_rank, world = dist_env()
    import fp8_paged_attention_gb300 as fp8pa  # the CUDA library; raises if it cannot load
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    w = synth.make_combine_config(args.config, device=dev)
    P, T, hq, d = w.o_parts.shape
    work = w.bytes_algorithmic()
    out = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((hq, T), dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        fp8pa.lse_combine(w.o_parts, w.lse_parts, out=out, lse=lse)
    torch.cuda.synchronize()
    ms_total, k_avg_ms, k_ev_ms, clock_info = time_single_launch(
        lambda i: fp8pa.lse_combine(w.o_parts, w.lse_parts, out=out, lse=lse), 0, args.steps, stream, world, dev,
        local_rank)
    peaks = measured_peaks()
    achieved = work / (k_avg_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": round(peaks["hbm_gbs"], 1), "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": ncu_traffic(w.name, COMBINE_SOURCES),
                "kernel": "lse_combine_kernel", "kernel_ms": round(k_avg_ms, 5),
                "kernel_ms_source": "mean over the timed region's back-to-back launches",
                "kernel_ms_events_per_launch": round(k_ev_ms, 5),
                "frac_events_per_launch": round(work / (k_ev_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "peak_source": peaks["source"] + " MEASURED_PEAKS.json hbm_gbs (copy)"}
    e2e = None
    if not args.no_e2e:
        h_o, h_l = w.o_parts.cpu().pin_memory(), w.lse_parts.cpu().pin_memory()
        h_out, h_lse = torch.empty(out.shape, dtype=out.dtype).pin_memory(), torch.empty(lse.shape).pin_memory()
        d_o, d_l = torch.empty_like(w.o_parts), torch.empty_like(w.lse_parts)

        def e2e_step():
            d_o.copy_(h_o, non_blocking=True)
            d_l.copy_(h_l, non_blocking=True)
            fp8pa.lse_combine(d_o, d_l, out=out, lse=lse)
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(10, args.steps // 10)
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e.record(stream)
        torch.cuda.synchronize()
        e_ms = slowest_rank_ms(a.elapsed_time(e), world, dev)
        e2e = {"value": round(job_rate(work, world, n_e2e, e_ms, False), 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h_o.numel() * 2 + h_l.numel() * 4),
               "d2h_bytes_per_step": int(h_out.numel() * 2 + h_lse.numel() * 4), "steps": n_e2e,
               "ms_per_step": round(e_ms / n_e2e, 5)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r, cores, desc, _t = combine_oracle_timing(synth.make_combine_config(args.config), args.cpu_budget)
        cpu = {"value": round(r, 6), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": round(job_rate(work, world, args.steps, ms_total, False), 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_total / args.steps, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "parts": P, "total_q": T, "num_heads_q": hq, "head_dim": d,
                       "bytes_per_step": work, "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {work / 1e6:.0f} MB per step"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clock_info}))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG,
                    choices=synth.CONFIG_NAMES + synth.KV_WRITE_CONFIG_NAMES + synth.COMBINE_CONFIG_NAMES)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ctas-per-sm", type=int, default=0, help="force 1 or 2 attention CTAs per SM (0 = auto)")
    ap.add_argument("--num-splits", type=int, default=0, help="split-KV count (0 = automatic)")
    ap.add_argument("--sinks", action="store_true", help="attention sinks, one logit per query head")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only --config (by default a one-GPU run also measures the other workloads)")
    ap.add_argument("--per-config-steps", type=int, default=0, help="timed steps per extra workload (0 = --steps)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.config in synth.KV_WRITE_CONFIG_NAMES:
        return run_kv_write(args)
    if args.config in synth.COMBINE_CONFIG_NAMES:
        return run_combine(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
