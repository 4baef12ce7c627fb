"""Pipeline trace of the tensor-core verify kernel on one GPU.

Builds a copy of the library with -DVMLA_TRACE in a temporary directory (the
in-tree library is left as it is), runs one seeded workload, and prints from
the global-timer stamps of cluster 0:
  * the steady-state tile period and its parts (the score-MMA issuer's wait for
    its K stage and for a free S buffer, the MMAs themselves, the K load's
    latency from issue to full);
  * each unit boundary: the Q load of the next unit, the mixer's epilogue and
    the epilogue command's round trip.
With --time it instead times the verify kernel (library events, L2 flushed
before each call) for each forced piece count, which gives the cost of a work
unit from the slope of time against units per cluster.

    python -m speculative_decoding_mla_gb300.microbench.trace_pipeline long_185k --splits 9
    python -m speculative_decoding_mla_gb300.microbench.trace_pipeline long_185k --time 9 18 36 54
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
EVENTS, TILES = 32, 256


def _child(root: str, workload: str, splits: int) -> None:
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
    ap.add_argument("--child", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.child:
        _child(args.child, args.workload, args.splits)
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
                            "--child", tmp], cwd=tmp)
        if r.returncode != 0:
            raise SystemExit(r.returncode)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


if __name__ == "__main__":
    main()
