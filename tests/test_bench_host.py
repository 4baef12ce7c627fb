"""Host-side logic of bench.py without a GPU: algorithmic work counts, and the
multi-rank aggregation (max time over ranks, summed tokens) on two gloo ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from speculative_decoding_mla_gb300 import synth


def test_algorithmic_work_causal_and_tree():
    case = synth.make_case("w", [10, 3], [4, 2], num_heads=2, pool_slots=30, seed=1)
    nbytes, flops, tokens = bench.algorithmic_work(case)
    assert tokens == 14 + 5
    # visible pairs: sum_b Q_b * P_b + causal triangles
    V = (4 * 10 + 10) + (2 * 3 + 3)
    assert flops == 2 * 2 * (576 + 512) * V
    assert nbytes == (19 * 1156) + (6 * 2 * (1152 + 1024 + 4))
    tree = synth.make_case("t", [5], [6], num_heads=1, pool_slots=11, tree_depth=2, seed=2)
    depth = np.zeros(6, int)
    for i in range(1, 6):
        depth[i] = depth[tree.parent[i]] + 1
    _, flops_t, _ = bench.algorithmic_work(tree)
    assert flops_t == 2 * 1 * 1088 * (6 * 5 + int((depth + 1).sum()))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), VMLA_BENCH_BACKEND="gloo")
    r, local, w = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    mx, sm = bench.reduce_max_sum(1.0 + rank, 10.0 * (rank + 1), w)
    out[rank] = (mx, sm)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        assert out[rank] == (2.0, 30.0)


def test_single_rank_is_identity():
    assert bench.reduce_max_sum(3.5, 7.0, 1) == (3.5, 7.0)


def test_source_fingerprint_ignores_comments_only(tmp_path):
    base = "int a = 1;  // one\n\n// a note\nint b = a + 1;\n"
    comment_edit = "int a = 1;   // the first\n// another note\n\nint b = a + 1;\n"
    code_edit = "int a = 2;  // one\n\n// a note\nint b = a + 1;\n"
    paths = []
    for name, text in (("base.cu", base), ("comment.cu", comment_edit), ("code.cu", code_edit)):
        p = tmp_path / name
        p.write_text(text)
        paths.append(str(p))
    fp = [bench.source_fingerprint([p]) for p in paths]
    assert fp[0] == fp[1] and fp[0] != fp[2]
    # the committed traffic figures apply exactly when the profiled code is unchanged
    assert (bench.traffic_per_launch("long_185k") is not None) == (bench.source_fingerprint() ==
                                                                   bench.PROFILED_FINGERPRINT)


def test_roofline_picks_the_bound_of_the_work():
    peaks = {"bf16_tflops": 1912.5, "hbm_gbs": 6789.3, "source": "measured"}
    # 185k-key prefix, 16 drafts, 64 heads: about 1900 flop per byte, above the ridge
    r = bench.roofline_entry(412.24e9, 216.1e6, 0.3313, peaks)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 412.24e9 / 0.3313e-3 / 1e12) < 1e-9 and abs(r["frac"] - r["achieved"] / 1912.5) < 1e-12
    # one draft per sequence: about 120 flop per byte, below the ridge, so the HBM copy rate bounds it
    r = bench.roofline_entry(89.23e9, 745.1e6, 0.3359, peaks)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 745.1e6 / 0.3359e-3 / 1e9) < 1e-9 and abs(r["frac"] - r["achieved"] / 6789.3) < 1e-12


def test_side_leg_records_a_failure_in_its_place():
    assert bench.side_leg(lambda a, b: {"ms": a + b}, 1, 2) == {"ms": 3}

    def broken():
        raise RuntimeError("device-planned call: bad shape")
    assert bench.side_leg(broken) == {"error": "RuntimeError: device-planned call: bad shape"}
