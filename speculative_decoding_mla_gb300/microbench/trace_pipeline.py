"""Pipeline trace of the tensor-core verify kernel on one GPU.

Builds a copy of the library with -DVMLA_TRACE in a temporary directory (the
in-tree library is left as it is), runs one seeded workload, and prints from
the global-timer stamps of cluster 0:
  * the steady-state tile period and its parts (the score-MMA issuer's wait for
    its K stage and for a free S buffer, the MMAs themselves, the K load's
    latency from issue to full);
  * each unit boundary: the Q load of the next unit, the mixer's epilogue and
    the epilogue command's round trip;
  * per cluster: its units and tiles, when it entered, finished its set-up,
    passed the wait for the previous launch, wrote its last outputs and left,
    which shows how evenly the schedule's work ends across the clusters.
With --time it instead times the verify kernel (library events, L2 flushed
before each call) for each forced piece count, which gives the cost of a work
unit from the slope of time against units per cluster.

    python -m speculative_decoding_mla_gb300.microbench.trace_pipeline long_185k --splits 9
    python -m speculative_decoding_mla_gb300.microbench.trace_pipeline long_185k --time 9 18 36 54
    python -m speculative_decoding_mla_gb300.microbench.trace_pipeline contiguous_1k --timeline

--timeline adds cluster 0's stamps of its first three and last two tiles (and
of the messages of those tiles), in microseconds from the earliest stamp.
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)

# trace event ids of the kernel (-DVMLA_TRACE); per tile unless noted
EV_K_ISSUE, EV_K_FULL, EV_S_FREE, EV_MMA_DONE = 0, 1, 12, 2
EV_Q_START, EV_Q_DONE, EV_EPI_START, EV_EPI_END, EV_CMD_POST, EV_CMD_DONE = 20, 21, 22, 23, 24, 25  # per unit
# per cluster (indexed by the cluster): stamps, and the count word units << 32 | tiles
EV_CL_ENTER, EV_CL_SETUP, EV_CL_DEP, EV_CL_LAST_OUT, EV_CL_EXIT, EV_CL_COUNTS = 26, 27, 28, 29, 30, 31
# what each per-tile (or per-message, per-unit) stamp of cluster 0 marks
TIMELINE = {
    0: "scorer 0: K load issued", 10: "scorer 1: K load issued", 1: "score MMAs: K stage full",
    12: "score MMAs: S buffer free", 2: "score MMAs issued", 3: "softmax 0: S full", 11: "softmax 1: S full",
    14: "softmax 0: first message's row maxima met", 15: "softmax 1: first message's row maxima met",
    4: "sender 0: slot free, message 0", 16: "sender 0: slot free, message 1",
    18: "sender 1: slot free, message 0", 17: "sender 1: slot free, message 1",
    5: "mixer 2: V load issued (per message)", 6: "PV MMAs: V stage full, message 0",
    7: "PV MMAs: P full, message 0", 19: "PV MMAs: P full, message 1", 8: "PV MMAs of the tile issued",
    13: "relay 3: message forwarded (per message)", 9: "release 2: message's products done (per message)",
}
UNIT_EVENTS = {20: "softmax 0: Q awaited", 21: "softmax 0: Q in TMEM", 22: "epilogue starts",
               23: "epilogue stored", 24: "epilogue command posted", 25: "epilogue command done"}
PER_MESSAGE = {5, 13, 9}
EVENTS, TILES = 32, 256


def _child(root: str, workload: str, splits: int, timeline: bool) -> None:
    import ctypes

    import numpy as np
    import torch

    sys.path.insert(0, root)
    from speculative_decoding_mla_gb300 import binding, device, synth

    lib = binding.lib()
    case = synth.workload(workload)
    dc = device.to_device(case, device="cuda:0")
    out, lse = device.alloc_outputs(dc)
    ws = device.alloc_workspace(dc, splits)
    info, per = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_TC, case.qo_indptr, case.kv_indptr, case.num_heads,
                                             splits)
    for _ in range(3):
        device.run(dc, kernel="tc", splits=splits, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    if lib.vmla_trace_clear() != 0:
        raise RuntimeError("trace buffer not cleared")
    device.run(dc, kernel="tc", splits=splits, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    status = binding.verify_attn_mla_check(ws)
    buf = (ctypes.c_uint64 * (EVENTS * TILES))()
    if lib.vmla_trace_read(buf, EVENTS * TILES) != EVENTS * TILES:
        raise RuntimeError("trace buffer not read")
    a = np.frombuffer(buf, dtype=np.uint64).reshape(EVENTS, TILES).astype(np.int64)
    counts = a[EV_CL_COUNTS].copy()
    a[EV_CL_COUNTS] = 0
    t0 = a[a > 0].min()
    us = np.where(a > 0, (a - t0) / 1e3, np.nan)
    # tiles of cluster 0's units, to leave out the first and last tile of each
    units = int(np.sum(~np.isnan(us[EV_Q_START])))
    edge = set()
    n_tiles = int(np.sum(~np.isnan(us[EV_MMA_DONE])))
    done = us[EV_MMA_DONE][:n_tiles]
    gaps = np.diff(done)
    med = float(np.nanmedian(gaps))
    for i, g in enumerate(gaps):
        if g > 3 * med:  # a unit boundary lies between tile i and i + 1
            edge |= {i, i + 1, i + 2}
    steady = [t for t in range(2, n_tiles) if t not in edge]

    def med_of(f):
        v = [f(t) for t in steady]
        v = [x for x in v if not np.isnan(x)]
        return round(float(np.median(v)), 3) if v else None

    res = {
        "workload": workload, "splits": splits, "units_total": int(info.num_units), "status": int(status),
        "cluster0_units": units, "cluster0_tiles": n_tiles,
        "tile_period_us": med_of(lambda t: done[t] - done[t - 1]),
        "k_load_latency_us": med_of(lambda t: us[EV_K_FULL][t] - us[EV_K_ISSUE][t]),
        "wait_k_us": med_of(lambda t: us[EV_K_FULL][t] - done[t - 1]),
        "wait_s_free_us": med_of(lambda t: us[EV_S_FREE][t] - us[EV_K_FULL][t]),
        "score_mma_us": med_of(lambda t: done[t] - us[EV_S_FREE][t]),
        "boundaries": [],
    }
    for u in range(units):
        res["boundaries"].append({
            "unit": u,
            "q_load_us": round(float(us[EV_Q_DONE][u] - us[EV_Q_START][u]), 2),
            "epilogue_us": round(float(us[EV_EPI_END][u] - us[EV_EPI_START][u]), 2),
            "epilogue_command_us": round(float(us[EV_CMD_DONE][u] - us[EV_CMD_POST][u]), 2),
        })
    res["boundary_mma_gaps_us"] = [round(float(g), 2) for g in gaps if g > 3 * med]
    n_cl = min(int(lib.vmla_trace_clusters()), TILES)
    clusters = []
    for c in range(n_cl):
        if np.isnan(us[EV_CL_ENTER][c]):
            continue
        clusters.append({
            "cluster": c, "units": int(counts[c] >> 32), "tiles": int(counts[c] & 0xFFFFFFFF),
            "enter_us": round(float(us[EV_CL_ENTER][c]), 2), "setup_us": round(float(us[EV_CL_SETUP][c]), 2),
            "dep_wait_us": round(float(us[EV_CL_DEP][c]), 2), "last_out_us": round(float(us[EV_CL_LAST_OUT][c]), 2),
            "exit_us": round(float(us[EV_CL_EXIT][c]), 2)})
    res["clusters"] = clusters
    if timeline:
        keep = [t for t in (0, 1, 2, n_tiles - 2, n_tiles - 1) if 0 <= t < n_tiles]
        keep = sorted(set(keep))
        rows = {}
        for ev, name in TIMELINE.items():
            if ev in PER_MESSAGE:
                idx = [2 * t + j for t in keep for j in (0, 1)]
            else:
                idx = keep
            rows[f"{ev:2d} {name}"] = [None if np.isnan(us[ev][i]) else round(float(us[ev][i]), 2) for i in idx]
        for ev, name in UNIT_EVENTS.items():
            rows[f"{ev:2d} {name}"] = [None if np.isnan(us[ev][u]) else round(float(us[ev][u]), 2)
                                       for u in range(units)]
        res["timeline_tiles"] = keep
        res["timeline"] = rows
    if clusters:
        ex = np.array([c["exit_us"] for c in clusters])
        work = [c for c in clusters if c["tiles"] > 0]
        res["cluster_summary"] = {
            "clusters_with_work": len(work), "exit_min_us": float(ex.min()), "exit_median_us": float(np.median(ex)),
            "exit_max_us": float(ex.max()),
            "latest": max(clusters, key=lambda c: c["exit_us"]),
            "tiles_min_max": [min(c["tiles"] for c in work), max(c["tiles"] for c in work)] if work else None,
        }
    print(json.dumps(res, indent=1))


def _time(workload: str, splits_list) -> None:
    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    from speculative_decoding_mla_gb300 import binding, build, device, synth

    build.build()
    case = synth.workload(workload)
    dc = device.to_device(case, device="cuda:0")
    out, lse = device.alloc_outputs(dc)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda:0")
    for sp in splits_list:
        ws = device.alloc_workspace(dc, sp)
        info, _ = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_TC, case.qo_indptr, case.kv_indptr,
                                               case.num_heads, sp)

        def step():
            flush.fill_(1)
            device.run(dc, kernel="tc", splits=sp, out=out, lse=lse, workspace=ws)

        for _ in range(4):
            step()
        torch.cuda.synchronize()
        binding.verify_attn_mla_timing_enable(15)
        for _ in range(15):
            step()
        torch.cuda.synchronize()
        _, v, m = binding.verify_attn_mla_timing_read(15)
        binding.verify_attn_mla_timing_enable(0)
        print(json.dumps({"workload": workload, "splits": sp, "units": int(info.num_units),
                          "status": int(binding.verify_attn_mla_check(ws)),
                          "verify_us": round(float(np.median(v)) * 1e3, 1),
                          "merge_us": round(float(np.median(m)) * 1e3, 1)}), flush=True)
        del ws


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("--splits", type=int, default=0, help="forced pieces per sequence (0: the planner's)")
    ap.add_argument("--time", type=int, nargs="*", help="time the verify kernel for these forced piece counts")
    ap.add_argument("--timeline", action="store_true", help="print cluster 0's stamps of its first and last tiles")
    ap.add_argument("--child", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.child:
        _child(args.child, args.workload, args.splits, args.timeline)
        return
    if args.time:
        _time(args.workload, args.time)
        return
    tmp = tempfile.mkdtemp(prefix="vmla_trace_")
    try:
        shutil.copytree(PKG, os.path.join(tmp, "speculative_decoding_mla_gb300"),
                        ignore=shutil.ignore_patterns("*.so", "__pycache__"))
        shutil.copytree(os.path.join(ROOT, "include"), os.path.join(tmp, "include"))
        import importlib.util

        # the copy's build module (its paths are relative to its own file)
        spec = importlib.util.spec_from_file_location(
            "vmla_trace_build", os.path.join(tmp, "speculative_decoding_mla_gb300", "build.py"))
        tbuild = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(tbuild)
        tbuild.build(force=True, extra_flags=("-DVMLA_TRACE",))
        r = subprocess.run([sys.executable, os.path.abspath(__file__), args.workload, "--splits", str(args.splits),
                            "--child", tmp] + (["--timeline"] if args.timeline else []), cwd=tmp)
        if r.returncode != 0:
            raise SystemExit(r.returncode)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


if __name__ == "__main__":
    main()
