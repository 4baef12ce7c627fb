#!/usr/bin/env python
"""Benchmark of the MLA speculative-decoding verify attention on GB300.

One step = one verify call (mask expansion when a tree is given, the KV row
gather, the verify kernel, the split merge) over one batch of seeded synthetic
inputs resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: long_185k (1 sequence, 185,000-token prefix + 16 causal draft
positions, 64 heads, 576-dim bf16 latent rows at page_size = 1 with permuted
slots in a 200,000-slot pool), the long-context shape of the pages' decode
workload.  Every workload whose KV rows are under twice the 129 MB L2 (this one's
are 213 MB) gets a 512 MB L2 flush before each step; larger ones need none.
Each step is timed between two CUDA events on the launching stream, recorded
after the flush and a synchronisation, so the step's time includes the host
planner, the launch gaps and every kernel; a second pass with the library's
per-kernel events gives the breakdown (kept out of the timed steps, where the
verify kernel starts under the gather's tail); a warm-L2 figure (no flush) is
reported beside it.

Metric: KV tokens per second (sum over sequences of N_b, per step), plus
algorithmic TFLOP/s and HBM GB/s.  Algorithmic work per launch:
  bytes = sum_b [N_b * (1152 + 4) + Q_b * H * (1152 + 1024 + 4)]
  flops = 2 * H * (576 + 512) * V,   V = sum_b (Q_b * P_b + sum_i |mask_i|)
Roofline: the verify kernel's achieved rate (algorithmic work / its mean
event-timed duration) against the roof that bounds the work: TFLOP/s against the
measured dense bf16 peak when the flops take longer there than the bytes at the
measured HBM copy rate, GB/s against that copy rate otherwise.

--impl reference times the CPU fp64 oracle on the host cores on a bounded
sample of the same workload (a subset of query rows), scaled to the metric.
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path shards by sequence with no exchange), value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-attn KV tokens/sec, TFLOPS and HBM GB/s as % of GB300 roofline"

# DRAM bytes (read + write) per verify launch from committed ncu captures of each workload's
# first timed launch; valid only while the kernel and planner sources are the ones profiled.
PROFILED_SOURCES = ("speculative_decoding_mla_gb300/csrc/vmla_tc.cu", "speculative_decoding_mla_gb300/csrc/vmla_plan.cpp",
                    "speculative_decoding_mla_gb300/csrc/vmla_plan_core.h")
PROFILED_FINGERPRINT = "08ef17040dd4e9d0"
PROFILED_TRAFFIC = {"contiguous_1k": 2.48e6, "paged_ragged": 80.57e6, "long_185k": 218.44e6, "tree_32k": 1303.96e6,
                    "sweep_q1": 754.48e6, "sweep_q4": 771.65e6, "sweep_q16": 826.08e6}


def source_fingerprint(paths=None) -> str:
    """First 16 hex digits of the sha256 of the profiled sources' code (or of `paths`): each line
    cut at `//`, trailing blanks and empty lines dropped, so that comment edits keep the fingerprint."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths if paths is not None else PROFILED_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def traffic_per_launch(workload: str):
    if source_fingerprint() != PROFILED_FINGERPRINT:
        return None
    return PROFILED_TRAFFIC.get(workload)
L2_BYTES = 129 * 1024 * 1024


def algorithmic_work(case):
    """(bytes, flops, kv_tokens) of one call, from the shapes and visibility counts."""
    H = case.num_heads
    nkv = np.diff(case.kv_indptr).astype(np.int64)
    nq = np.diff(case.qo_indptr).astype(np.int64)
    prefix = nkv - nq
    vis_draft = 0
    for b in range(case.batch):
        n = int(nq[b])
        if case.parent is None:
            vis_draft += n * (n + 1) // 2
        else:
            par = case.parent[case.qo_indptr[b]:case.qo_indptr[b + 1]]
            depth = np.zeros(n, np.int64)
            for i in range(n):
                depth[i] = 0 if par[i] < 0 else depth[par[i]] + 1
            vis_draft += int((depth + 1).sum())
    V = int((nq * prefix).sum()) + vis_draft
    bytes_ = int((nkv * (1152 + 4)).sum() + (nq * H * (1152 + 1024 + 4)).sum())
    flops = 2 * H * (576 + 512) * V
    return bytes_, flops, int(nkv.sum())


def side_leg(fn, *args):
    """One of the measurements printed beside the step (other entry points on the same workload);
    a failure there is recorded in its place instead of costing the step's line."""
    try:
        return fn(*args)
    except Exception as e:  # noqa: BLE001 -- reported in the JSON line
        return {"error": f"{type(e).__name__}: {e}"}


def roofline_entry(flops: float, nbytes: float, kernel_ms: float, peaks: dict) -> dict:
    """The verify kernel against the roof that bounds its algorithmic work: the dense bf16 tensor
    peak when the flops take longer there than the bytes at the HBM copy rate (many draft rows per
    key), the HBM copy rate otherwise (one or few draft rows per key)."""
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = flops / (kernel_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "peak_source": f"{peaks['source']} dense bf16 burst"}
    achieved = nbytes / (kernel_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} HBM copy"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.25)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        mhz, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not mhz:
            return None
        return {"sm_mhz": float(np.median(mhz)), "sm_max_mhz": float(max(maxes)), "reasons": sorted(reasons),
                "samples": len(mhz)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("VMLA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def reduce_max_sum(value_max: float, value_sum: float, world: int, device=None):
    """(max over ranks of value_max, sum over ranks of value_sum); identity when world == 1."""
    if world <= 1:
        return value_max, value_sum
    import torch
    import torch.distributed as dist
    t1 = torch.tensor([value_max], dtype=torch.float64, device=device)
    t2 = torch.tensor([value_sum], dtype=torch.float64, device=device)
    dist.all_reduce(t1, op=dist.ReduceOp.MAX)
    dist.all_reduce(t2, op=dist.ReduceOp.SUM)
    return float(t1.item()), float(t2.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_oracle_sample(case, budget_s: float = 15.0, max_rows: int = 4096):
    """Times the oracle on a growing sample of rows; returns (kv tokens/s, cores, sample text)."""
    import oracle
    H = case.num_heads
    T = case.q.shape[0]
    total_rows = T * H
    cores = oracle.num_cpus()
    # KV keys each row reads (its sequence's N_b)
    nkv = np.diff(case.kv_indptr).astype(np.int64)
    seq_of_t = np.repeat(np.arange(case.batch), np.diff(case.qo_indptr))
    keys_per_row = np.repeat(nkv[seq_of_t], H)
    rng_rows = synth_rows(total_rows)
    n = min(total_rows, max(cores, 16))
    spent = 0.0
    done_rows = 0
    done_keys = 0
    while True:
        rows = rng_rows[done_rows:done_rows + n]
        if len(rows) == 0:
            break
        t0 = time.perf_counter()
        oracle.verify_rows(case, rows)
        dt = time.perf_counter() - t0
        spent += dt
        done_rows += len(rows)
        done_keys += int(keys_per_row[rows].sum())
        if spent >= budget_s or done_rows >= min(total_rows, max_rows):
            break
        # next batch: most of the remaining budget at the last batch's rate, at most 4x that batch
        # (small batches are dominated by thread start-up); stop when less than a batch of one row
        # per core still fits
        n = int(min(total_rows - done_rows, 4 * len(rows), 0.8 * (budget_s - spent) * len(rows) / max(dt, 1e-3)))
        if n < cores:
            break
    # whole-job time estimate: (all rows' keys) / (keys per second achieved on the sample)
    keys_per_s = done_keys / spent
    all_keys = int(keys_per_row.sum())
    job_s = all_keys / keys_per_s
    tokens = int(nkv.sum())
    sample = f"{done_rows} of {total_rows} query rows (seeded), {spent:.1f} s of CPU wall time, scaled by row keys"
    return tokens / job_s, cores, sample, spent


def synth_rows(total_rows: int) -> np.ndarray:
    from speculative_decoding_mla_gb300 import synth
    w = synth.words(17, synth.TAG_AUX, total_rows)
    return np.argsort(w, kind="stable").astype(np.int64)


def run_reference(args, rank, world):
    from speculative_decoding_mla_gb300 import synth
    if rank != 0:
        barrier(world)
        return
    case = synth.workload(args.workload)
    per_step = max(1.0, args.ref_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        cpu_oracle_sample(case, budget_s=0.5, max_rows=16)
    vals = []
    total_s = 0.0
    for _ in range(args.steps):
        v, cores, sample, spent = cpu_oracle_sample(case, budget_s=per_step)
        vals.append(v)
        total_s += spent
    value = float(np.median(vals))
    nbytes, flops, tokens = algorithmic_work(case)
    ms = tokens / value * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded splitmix64/Box-Muller, bf16 inputs)",
        "config": {"workload": args.workload, "heads": case.num_heads, "batch": case.batch,
                   "kv_tokens": tokens, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "KV tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {sample}"},
        "e2e": {"value": value, "unit": "KV tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    barrier(world)


def run_ours(args, rank, local, world):
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    if not os.path.exists(os.path.join(ROOT, "speculative_decoding_mla_gb300", "libvmla.so")):
        vbuild.build()
    from speculative_decoding_mla_gb300 import binding, device, synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    case = synth.workload(args.workload)
    dc = device.to_device(case, device=dev)
    out, lse = device.alloc_outputs(dc)
    ws = device.alloc_workspace(dc, args.splits)
    nbytes, flops, tokens = algorithmic_work(case)
    input_bytes = int(case.kv_indices.max() + 1) * 1152 if case.batch else 0
    flush = input_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None
    stream = torch.cuda.current_stream(dev)
    kernel = "simt" if args.kernel == "simt" else "tc"

    # the call, its arguments checked and marshalled once (binding.prepare_verify_attn_mla)
    call = binding.prepare_verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                           dc.kv_indptr_host, dc.qo_indptr_host, out, lse, ws, dc.sm_scale,
                                           draft_mask=dc.draft_mask, parent=dc.parent, splits=args.splits,
                                           stream=stream, kernel=kernel)

    def step():
        if flush_buf is not None:
            flush_buf.fill_(1)
        call()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    st = binding.verify_attn_mla_check(ws)
    if st != 0:
        raise RuntimeError(f"kernel status {binding.status_string(st)}")

    # Each step is timed between two events on the launching stream, from an idle
    # GPU: the L2 flush and a synchronisation come before the first event, so the
    # host planner, the launch gaps and every kernel of the call fall inside.
    def timed_steps(steps):
        events = []
        for _ in range(steps):
            if flush_buf is not None:
                flush_buf.fill_(1)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            events.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in events]))

    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    step_ms = timed_steps(args.steps)
    barrier(world)
    clocks = sampler.stop()
    # The per-kernel breakdown from the same steps run again with the library's
    # events around each kernel (kept out of the timed steps above: an event
    # between two kernels keeps the second from starting under the first's tail).
    binding.verify_attn_mla_timing_enable(args.steps)
    timed_steps(args.steps)
    gather_ms, verify_ms, merge_ms = binding.verify_attn_mla_timing_read(args.steps)
    binding.verify_attn_mla_timing_enable(0)
    kernel_ms = float(gather_ms.mean() + verify_ms.mean() + merge_ms.mean())
    max_ms, sum_tokens = reduce_max_sum(step_ms, float(tokens), world, dev if world > 1 else None)
    value = sum_tokens / (max_ms / 1e3)
    st = binding.verify_attn_mla_check(ws)
    if st != 0:
        raise RuntimeError(f"kernel status {binding.status_string(st)}")

    # the same step with the inputs left warm in L2 (no flush, back to back)
    warm_events = []
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        warm_events.append((e0, e1))
    torch.cuda.synchronize()
    warm_ms = float(np.mean([a.elapsed_time(b) for a, b in warm_events]))

    # end to end through the host-buffer entry point: H2D of the step's inputs,
    # the call, D2H of out and lse, synchronised, wall clock
    T, H = case.q.shape[0], case.num_heads
    q_h = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    kvi_h = torch.from_numpy(case.kv_indices).pin_memory()
    out_h = torch.empty((T, H, 512), dtype=torch.int16).pin_memory()
    lse_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    par_h = torch.from_numpy(case.parent).pin_memory() if case.parent is not None else None
    nbuf = binding.verify_attn_mla_host_buffer_size(case.qo_indptr, case.kv_indptr, H, args.splits,
                                                    has_parent=par_h is not None)
    dbuf = torch.empty(nbuf, dtype=torch.uint8, device=dev)

    e2e_step = binding.prepare_verify_attn_mla_host(q_h, dc.kv_pool, case.kv_indptr, kvi_h, case.qo_indptr, out_h,
                                                    lse_h, dbuf, case.sm_scale, parent_host=par_h,
                                                    splits=args.splits, stream=stream)

    for _ in range(3):
        e2e_step()
    barrier(world)
    e2e_total = 0.0
    for _ in range(args.steps):
        if flush_buf is not None:  # the flush is not part of the step: outside the timed region
            flush_buf.fill_(1)
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()  # returns once out and lse are in host memory
        e2e_total += time.perf_counter() - t0
    e2e_s = e2e_total / args.steps
    e2e_max, e2e_tokens = reduce_max_sum(e2e_s, float(tokens), world, dev if world > 1 else None)
    # bytes that cross to the device: q, the indices (read in place by the gather, being page-locked)
    # and, for a tree, its parents and qo_indptr; kv_indptr is read on the host for the plan only
    h2d = q_h.numel() * 2 + kvi_h.numel() * 4 + ((par_h.numel() + case.batch + 1) * 4 if par_h is not None else 0)
    d2h = out_h.numel() * 2 + lse_h.numel() * 4

    # the stream-capture-safe entry point (plan computed on the device) captured
    # once in a CUDA graph and replayed on the same workload, one replay per step
    graph = side_leg(device_plan_graph, args, case, dc, stream, flush_buf, tokens)
    accept = side_leg(tree_accept_timing)
    runs = side_leg(defragmented_runs, args, case, dc, flush_buf, tokens)
    fp8 = side_leg(fp8_pool_timing, args, case, dc, flush_buf, tokens)

    peaks = load_peaks()
    v_ms = float(verify_ms.mean())
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, spent = cpu_oracle_sample(case, budget_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "KV tokens/s", "cores": cores, "kind": "oracle", "sample": sample}
    launches_per_step = (1 + (1 if float(merge_ms.max()) > 0 else 0) + (1 if float(gather_ms.max()) > 0 else 0)
                         + (1 if case.parent is not None else 0))
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded splitmix64/Box-Muller, bf16 inputs)",
            "config": {"workload": args.workload, "batch": case.batch, "heads": H, "kv_tokens": tokens,
                       "draft_tokens": T, "kernel": kernel, "splits": args.splits or "auto",
                       "l2": "flushed (512 MB write) before every step" if flush_buf is not None
                       else "inputs larger than L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "tflops": flops / (max_ms / 1e3) / 1e12,
            "hbm_gbs": nbytes / (max_ms / 1e3) / 1e9,
            "roofline": dict(roofline_entry(flops, nbytes, v_ms, peaks),
                             traffic=traffic_per_launch(args.workload), kernel="verify",
                             algorithmic_flops=flops, algorithmic_bytes=nbytes, verify_ms=v_ms,
                             merge_ms=float(merge_ms.mean()), gather_ms=float(gather_ms.mean()),
                             roofline_ms=max(flops / (peaks["bf16_tflops"] * 1e12),
                                             nbytes / (peaks["hbm_gbs"] * 1e9)) * 1e3),
            "roofline_frac_step": max(flops / (peaks["bf16_tflops"] * 1e12),
                                      nbytes / (peaks["hbm_gbs"] * 1e9)) * 1e3 / max_ms,
            "step_breakdown_ms": {"gather": float(gather_ms.mean()), "verify": float(verify_ms.mean()),
                                  "merge": float(merge_ms.mean()), "kernels": kernel_ms,
                                  "planner_gaps_and_overlap": step_ms - kernel_ms,
                                  "note": "kernel times from a second pass with an event around each kernel; "
                                          "in the timed steps the verify kernel starts under the gather's tail "
                                          "and the merge under the verify's"},
            "warm_l2": {"ms_per_step": warm_ms, "value": tokens / (warm_ms / 1e3), "unit": "KV tokens/s",
                        "note": "same call back to back, no flush between steps"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_tokens / e2e_max, "unit": "KV tokens/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "note": "every step q crosses in from pinned host memory, the pinned indices are read in place "
                            "by the gather (and a tree's parents and qo_indptr are copied), out and lse are copied "
                            "back; the KV cache stays resident in HBM"},
            "gpu_launches": int(launches_per_step * args.steps),
            "device_plan_graph": graph,
            "tree_accept": accept,
            "defragmented": runs,
            "fp8_kv": fp8,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def timed_from_idle(call, steps, flush_buf, stream=None):
    """Mean ms of `call` between two events on `stream`, each step from an idle GPU (the L2 flush and a
    synchronisation come before the first event), as the main step is timed: the host work of the
    call, its launch gaps and every kernel fall inside."""
    import torch
    stream = stream if stream is not None else torch.cuda.current_stream()
    events = []
    for _ in range(steps):
        if flush_buf is not None:
            flush_buf.fill_(1)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        events.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in events]))


def defragmented_runs(args, case, dc, flush_buf, tokens):
    """Defragments the workload's rows once into 128-aligned pool runs, then times the verify call on the runs."""
    import torch
    from speculative_decoding_mla_gb300 import binding
    n = np.diff(case.kv_indptr).astype(np.int64)
    padded = (n + 127) // 128 * 128
    base = np.zeros(case.batch, np.int64)
    base[1:] = np.cumsum(padded)[:-1]
    slots = int(padded.sum())
    dst = torch.empty((max(slots, 1), 576), dtype=torch.bfloat16, device=dc.q.device)
    base_d = torch.from_numpy(base.astype(np.int32)).to(dc.q.device)
    st = torch.zeros(2, dtype=torch.int32, device=dc.q.device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    binding.verify_attn_mla_defrag(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, dst, base_d, st)
    e1.record()
    torch.cuda.synchronize()
    defrag_ms = e0.elapsed_time(e1)
    if int(st[0]) != 0:
        raise RuntimeError(f"defragmentation: {binding.status_string(int(st[0]))}")
    out = torch.empty((dc.total_q, dc.num_heads, 512), dtype=torch.bfloat16, device=dc.q.device)
    lse = torch.empty((dc.total_q, dc.num_heads), dtype=torch.float32, device=dc.q.device)
    ws = torch.empty(binding.verify_attn_mla_runs_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host, dc.num_heads,
                                                                 args.splits), dtype=torch.uint8, device=dc.q.device)

    call = binding.prepare_verify_attn_mla_runs(dc.q, dst, dc.kv_indptr, base_d, dc.qo_indptr, dc.kv_indptr_host,
                                                dc.qo_indptr_host, out, lse, ws, dc.sm_scale, parent=dc.parent,
                                                splits=args.splits)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    ms = timed_from_idle(call, args.steps, flush_buf)
    status = binding.verify_attn_mla_check(ws)
    if status != 0:
        raise RuntimeError(f"verify on runs: {binding.status_string(status)}")
    # a decode loop keeps the runs: each step appends only its new rows (here the drafts, the
    # last Q_b rows of every sequence) and then verifies on the runs; timed as one event pair
    nq = np.diff(case.qo_indptr).astype(np.int64)
    first = torch.from_numpy((n - nq).astype(np.int32)).to(dc.q.device)

    append = binding.prepare_verify_attn_mla_defrag_append(dc.kv_pool, dc.kv_indptr, dc.kv_indices,
                                                           dc.kv_indptr_host, dst, base_d, first, st,
                                                           max_new_rows=int(nq.max()))

    def decode_step():
        append()
        call()

    for _ in range(max(3, args.warmup)):
        decode_step()
    torch.cuda.synchronize()
    dms = timed_from_idle(decode_step, args.steps, flush_buf)
    if int(st[0]) != 0 or binding.verify_attn_mla_check(ws) != 0:
        raise RuntimeError("decode step on runs reported a fault")
    # the same decode step captured once in a CUDA graph: the append with a bound and the call on
    # the runs with the plan made on the device, so that replays stay valid as the lengths change
    T, H, N = dc.total_q, dc.num_heads, int(case.kv_indptr[-1])
    gws = torch.empty(binding.verify_attn_mla_runs_device_plan_workspace_size(case.batch, H, T, N, args.splits),
                      dtype=torch.uint8, device=dc.q.device)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        binding.verify_attn_mla_defrag_append(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, dst,
                                              base_d, first, st, max_new_rows=int(nq.max()))
        binding.verify_attn_mla_runs_device_plan(dc.q, dst, dc.kv_indptr, base_d, dc.qo_indptr, case.batch, T, N,
                                                 out, lse, gws, dc.sm_scale, parent=dc.parent, splits=args.splits)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    gms = timed_from_idle(graph.replay, args.steps, flush_buf)
    if int(st[0]) != 0 or binding.verify_attn_mla_check(gws) != 0:
        raise RuntimeError("captured decode step on runs reported a fault")
    return {"ms_per_step": ms, "value": tokens / (ms / 1e3), "unit": "KV tokens/s", "defrag_ms_once": defrag_ms,
            "decode_step": {"ms_per_step": dms, "value": tokens / (dms / 1e3), "unit": "KV tokens/s",
                            "appended_rows_per_step": int(nq.sum()),
                            "note": "verify_attn_mla_defrag_append of the step's new rows (the drafts) into the "
                                    "runs, then verify_attn_mla_runs; one event pair per step from an idle GPU"},
            "decode_step_graph": {"ms_per_step": gms, "value": tokens / (gms / 1e3), "unit": "KV tokens/s",
                                  "note": "the decode step captured once in a CUDA graph (append with a bound, then "
                                          "verify_attn_mla_runs_device_plan); one replay per step from an idle GPU"},
            "note": "rows compacted once into 128-aligned pool runs (verify_attn_mla_defrag), then "
                    "verify_attn_mla_runs each step: no per-call gather; one event pair per call from an idle "
                    "GPU, as the main step"}


def fp8_pool_timing(args, case, dc, flush_buf, tokens):
    """The same workload with the latent pool stored as e4m3 codes and one scale (verify_attn_mla_fp8)."""
    import torch
    from speculative_decoding_mla_gb300 import binding
    vals = dc.kv_pool.float()
    scale = float(vals.abs().max()) / 400.0
    pool8 = (vals / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    del vals
    out = torch.empty((dc.total_q, dc.num_heads, 512), dtype=torch.bfloat16, device=dc.q.device)
    lse = torch.empty((dc.total_q, dc.num_heads), dtype=torch.float32, device=dc.q.device)
    ws = torch.empty(binding.verify_attn_mla_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host, dc.num_heads,
                                                            args.splits), dtype=torch.uint8, device=dc.q.device)

    call = binding.prepare_verify_attn_mla_fp8(dc.q, pool8, scale, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                               dc.kv_indptr_host, dc.qo_indptr_host, out, lse, ws, dc.sm_scale,
                                               parent=dc.parent, splits=args.splits)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    ms = timed_from_idle(call, args.steps, flush_buf)
    status = binding.verify_attn_mla_check(ws)
    if status != 0:
        raise RuntimeError(f"fp8 pool: {binding.status_string(status)}")
    return {"ms_per_step": ms, "value": tokens / (ms / 1e3), "unit": "KV tokens/s", "pool_bytes_per_key": 576,
            "note": "latent pool as e4m3 codes with one scale; the gather dequantizes into the bf16 staged rows; "
                    "one event pair per call from an idle GPU, as the main step"}


def tree_accept_timing(batch=32, nodes=64, calls=200):
    """Times the tree-acceptance kernel on seeded random trees of `nodes` drafts per sequence."""
    import torch
    from speculative_decoding_mla_gb300 import binding, synth
    rng = np.random.default_rng(5)
    qo = np.arange(batch + 1, dtype=np.int32) * nodes
    parent = np.concatenate([synth.tree_parents(5, nodes, 8, b) for b in range(batch)]).astype(np.int32)
    target = rng.integers(0, 8, batch * nodes).astype(np.int32)
    root = rng.integers(0, 8, batch).astype(np.int32)
    follow = np.where(parent < 0, root[np.arange(batch * nodes) // nodes], target[np.maximum(parent, 0) +
                                                                              (np.arange(batch * nodes) // nodes) * nodes])
    draft = np.where(rng.random(batch * nodes) < 0.8, follow, rng.integers(0, 8, batch * nodes)).astype(np.int32)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    qo_d, par_d, dr_d, tg_d, rt_d = d(qo), d(parent), d(draft), d(target), d(root)
    acc = torch.empty(batch, dtype=torch.int32, device="cuda")
    path = torch.empty(batch * nodes, dtype=torch.int32, device="cuda")
    nxt = torch.empty(batch, dtype=torch.int32, device="cuda")
    for _ in range(5):
        binding.verify_attn_mla_tree_accept(qo_d, par_d, dr_d, tg_d, rt_d, acc, path, nxt)
    torch.cuda.synchronize()
    # the calls are captured in one graph and replayed, so that the figure is the kernels' device time
    # and not the rate at which the host can issue them
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(calls):
            binding.verify_attn_mla_tree_accept(qo_d, par_d, dr_d, tg_d, rt_d, acc, path, nxt,
                                                stream=side.cuda_stream)
    graph.replay()
    torch.cuda.synchronize()
    per_call = []
    with torch.cuda.stream(side):  # the replay runs on the current stream: the events go on the same one
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(side)
            graph.replay()
            e1.record(side)
            torch.cuda.synchronize()
            per_call.append(e0.elapsed_time(e1) * 1e3 / calls)
    return {"us_per_call": float(np.median(per_call)), "batch": batch, "nodes_per_sequence": nodes,
            "mean_accepted": float(acc.float().mean()),
            "note": f"one warp per sequence; {calls} calls captured in a CUDA graph, median of 5 replays"}


def device_plan_graph(args, case, dc, stream, flush_buf, tokens):
    """Times graph replays of the device-planned call; returns a summary dict."""
    import torch
    from speculative_decoding_mla_gb300 import binding
    T, H, N = dc.total_q, dc.num_heads, int(case.kv_indptr[-1])
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=dc.q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=dc.q.device)
    ws = torch.empty(binding.verify_attn_mla_device_plan_workspace_size(case.batch, H, T, N, args.splits),
                     dtype=torch.uint8, device=dc.q.device)

    def call(s):
        binding.verify_attn_mla_device_plan(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, case.batch,
                                            T, N, out, lse, ws, dc.sm_scale, parent=dc.parent, splits=args.splits,
                                            stream=s)

    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call(side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(torch.cuda.current_stream())
    for _ in range(max(3, args.warmup)):
        g.replay()
    torch.cuda.synchronize()
    ms = timed_from_idle(g.replay, args.steps, flush_buf)
    st = binding.verify_attn_mla_check(ws)
    if st != 0:
        raise RuntimeError(f"device-planned call: {binding.status_string(st)}")
    return {"ms_per_step": ms, "value": tokens / (ms / 1e3), "unit": "KV tokens/s",
            "note": "verify_attn_mla_device_plan captured once in a CUDA graph (planner, mask, gather, verify and "
                    "merge kernels), one replay per step from an idle GPU, inputs resident in HBM"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_185k")
    ap.add_argument("--kernel", default="tc", choices=["tc", "simt"])
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    rank, local, world = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
