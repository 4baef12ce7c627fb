"""GPU tests of the device-planned (stream-capture-safe) entry point: its
results equal the host-planned call's bit for bit (both cut the same pieces),
and one captured CUDA graph replayed with other lengths, indices and contents
matches the oracle each time; lengths past the bounds are refused on the
device."""
import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth
from tests.test_gpu_parity import compare, run_full, small

pytestmark = pytest.mark.gpu


def _mods():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding, device
    return torch, binding, device


def run_dplan(case, splits=0, slack_q=0, slack_kv=0):
    """One device-planned call on buffers sized for the case plus slack; returns (out, lse, status)."""
    torch, binding, device = _mods()
    dc = device.to_device(case)
    T, H = dc.total_q, dc.num_heads
    maxq, maxkv = T + slack_q, int(case.kv_indptr[-1]) + slack_kv
    q = torch.zeros((max(maxq, 1), H, 576), dtype=torch.bfloat16, device="cuda")
    q[:T] = dc.q
    kvi = torch.zeros(max(maxkv, 1), dtype=torch.int32, device="cuda")
    kvi[:dc.kv_indices.numel()] = dc.kv_indices
    out = torch.full((max(maxq, 1), H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((max(maxq, 1), H), float("nan"), dtype=torch.float32, device="cuda")
    n = binding.verify_attn_mla_device_plan_workspace_size(case.batch, H, maxq, maxkv, splits)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_device_plan(q, dc.kv_pool, dc.kv_indptr, kvi, dc.qo_indptr, case.batch, maxq, maxkv,
                                        out, lse, ws, dc.sm_scale, parent=dc.parent, splits=splits)
    st = binding.verify_attn_mla_check(ws)
    torch.cuda.synchronize()
    return device.bf16_to_f64(out[:T]), lse[:T].cpu().numpy().astype(np.float64), st


@pytest.mark.parametrize("name", ["one_seq", "ragged", "tree", "heads_odd", "decode_q1"])
def test_device_plan_equals_host_plan_bitwise(name):
    case = small(name, seed=410)
    o1, l1, s1 = run_full(case, "tc")
    o2, l2, s2 = run_dplan(case, slack_q=5, slack_kv=300)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("splits", [1, 3, 7])
def test_device_plan_forced_splits_bitwise(splits):
    case = small("ragged", seed=411)
    o1, l1, _ = run_full(case, "tc", splits=splits)
    o2, l2, st = run_dplan(case, splits=splits)
    assert st == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_device_plan_contiguous_1k_against_oracle():
    case = synth.workload("contiguous_1k")
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_dplan(case)
    assert st == 0
    compare(o, l, ref_o, ref_l, "device plan / contiguous_1k")


def _step(name, prefixes, drafts, seed, H, pool):
    return synth.make_case(name, prefixes, drafts, num_heads=H, pool_slots=pool, seed=seed)


def test_captured_graph_replays_with_new_lengths():
    torch, binding, device = _mods()
    H, B, pool = 16, 3, 9000
    steps = [_step("a", [1000, 2000, 300], [16, 8, 4], 421, H, pool),
             _step("b", [700, 4100, 50], [4, 16, 12], 422, H, pool),
             _step("c", [0, 130, 5000], [1, 64, 2], 423, H, pool)]
    maxq = max(s.q.shape[0] for s in steps)
    maxkv = max(int(s.kv_indptr[-1]) for s in steps)
    q = torch.zeros((maxq, H, 576), dtype=torch.bfloat16, device="cuda")
    kv_pool = torch.zeros((pool, 576), dtype=torch.bfloat16, device="cuda")
    kvp = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    qop = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    kvi = torch.zeros(maxkv, dtype=torch.int32, device="cuda")
    out = torch.zeros((maxq, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((maxq, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.verify_attn_mla_device_plan_workspace_size(B, H, maxq, maxkv, 0), dtype=torch.uint8,
                     device="cuda")

    def load(case):
        dc = device.to_device(case)
        T, N = dc.total_q, dc.kv_indices.numel()
        q[:T].copy_(dc.q)
        kv_pool.copy_(dc.kv_pool)
        kvp.copy_(dc.kv_indptr)
        qop.copy_(dc.qo_indptr)
        kvi[:N].copy_(dc.kv_indices)
        torch.cuda.synchronize()
        return dc

    def call(stream):
        binding.verify_attn_mla_device_plan(q, kv_pool, kvp, kvi, qop, B, maxq, maxkv, out, lse, ws,
                                            steps[0].sm_scale, stream=stream)

    load(steps[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side)  # outside the capture: device set-up and the cluster count are looked up once
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(torch.cuda.current_stream())
    torch.cuda.synchronize()
    for case in steps:
        dc = load(case)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert binding.verify_attn_mla_check(ws) == 0
        T = dc.total_q
        o = device.bf16_to_f64(out[:T])
        l = lse[:T].cpu().numpy().astype(np.float64)
        ref_o, ref_l = oracle.verify(case)
        compare(o, l, ref_o, ref_l, f"graph replay {case.name}")
        o_host, l_host, _ = run_full(case, "tc")
        assert np.array_equal(o, o_host) and np.array_equal(l, l_host)
    # lengths past the bounds: nothing is computed and the status says why
    big = np.array(steps[1].kv_indptr, np.int32)
    big[-1] = maxkv + 1
    kvp.copy_(torch.from_numpy(big))
    out.fill_(0.5)
    g.replay()
    torch.cuda.synchronize()
    assert binding.verify_attn_mla_check(ws) == binding.VMLA_ERR_SHAPE
    assert bool(torch.all(out == 0.5))


@pytest.mark.slow
def test_device_plan_long_185k_sampled_rows():
    """The device-planned call on the full 185,000-token workload (the bench's graph-replayed path):
    bit-equal to the host-planned call, and sampled rows against the oracle."""
    from tests.test_gpu_parity import full_case, oracle_rows, sample_rows
    case = full_case("long_185k")
    o1, l1, s1 = run_full(case, "tc")
    o2, l2, s2 = run_dplan(case)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    rows = sample_rows(case)
    ref_o, ref_l = oracle_rows(case, rows, "long_185k/sampled")
    compare(o2.reshape(-1, o2.shape[-1])[rows], l2.reshape(-1)[rows], ref_o, ref_l, "device plan / long_185k")


def _random_batches():
    """Ragged batches on which the piece-size search leaves the default: lengths, drafts and heads
    drawn from a seeded generator (1 to 65 sequences; the last one above the search's 64)."""
    rng = np.random.default_rng(430)
    shapes = [(3, 64, [16, 4, 1], [30000, 500, 12000])]
    for B, H, dmax, med in [(12, 16, 64, 3000), (33, 64, 4, 4000), (64, 8, 64, 800), (5, 128, 8, 8000),
                            (65, 16, 16, 300)]:
        drafts = rng.integers(1, dmax + 1, B).tolist()
        prefixes = np.minimum(rng.lognormal(np.log(med), 1.0, B).astype(np.int64), 40000).tolist()
        shapes.append((B, H, drafts, prefixes))
    for i, (B, H, drafts, prefixes) in enumerate(shapes):
        nd = int(sum(drafts))
        yield synth.make_case(f"rand{i}", prefixes, drafts, num_heads=H,
                              pool_slots=int(sum(prefixes)) + nd + 64, seed=431 + i)


def test_device_plan_random_batches_bitwise():
    """The device planner scores the same piece-size candidates as the host planner (one warp per
    candidate), weighs the lane plan the same way, and must cut every sequence alike: bit-equal
    results on ragged random batches, and sampled rows of two of them against the oracle."""
    _, binding, _ = _mods()
    from tests.test_capi_cpu import _piece_rule
    from tests.test_gpu_parity import sample_rows
    changed = lanes = 0
    for k, case in enumerate(_random_batches()):
        o1, l1, s1 = run_full(case, "tc")
        o2, l2, s2 = run_dplan(case, slack_q=3, slack_kv=500)
        assert s1 == 0 and s2 == 0, case.name
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), case.name
        info, per = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_TC, case.qo_indptr, case.kv_indptr,
                                                 case.num_heads, 0, 144)
        default, _ = _piece_rule(case.qo_indptr, case.kv_indptr, case.num_heads, 36, search=False)
        changed += int([int(p) for p in per] != default)
        lanes += int(info.lane_width > 0)
        if k in (0, 2):
            rows = sample_rows(case, n=60, seed=k)
            ref_o, ref_l = oracle.verify_rows(case, rows)
            H = case.num_heads
            compare(o2.reshape(-1, o2.shape[-1])[rows], l2.reshape(-1)[rows], ref_o, ref_l, case.name)
    assert changed >= 1  # the search chose another piece size (or the lane plan) on some of these batches
    assert lanes >= 1  # and the lane plan on some


def test_length_error_wins_over_slot_error():
    """The gather starts beside the planner on the lengths it is given, so it may meet a slot outside
    the pool in entries the planner goes on to reject: the status word then says VMLA_ERR_SHAPE (the
    length error), and out and lse keep their contents.  With valid lengths the same bad slot is
    reported as VMLA_ERR_INDEX."""
    torch, binding, device = _mods()
    case = small("ragged", seed=840)
    dc = device.to_device(case)
    T, H, B = dc.total_q, dc.num_heads, case.batch
    maxq, maxkv = T, int(case.kv_indptr[-1])
    q = dc.q.clone()
    kvi = torch.full((maxkv,), case.pool_slots + 9, dtype=torch.int32, device="cuda")  # every slot outside
    out = torch.full((maxq, H, 512), 0.25, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((maxq, H), 0.25, dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.verify_attn_mla_device_plan_workspace_size(B, H, maxq, maxkv, 0), dtype=torch.uint8,
                     device="cuda")
    bad = np.array(case.kv_indptr, np.int32)
    bad[-1] = maxkv + 3  # past the bound: the planner refuses the lengths
    kvp_bad = torch.from_numpy(bad).cuda()
    binding.verify_attn_mla_device_plan(q, dc.kv_pool, kvp_bad, kvi, dc.qo_indptr, B, maxq, maxkv, out, lse, ws,
                                        dc.sm_scale)
    assert binding.verify_attn_mla_check(ws) == binding.VMLA_ERR_SHAPE
    assert bool(torch.all(out == 0.25)) and bool(torch.all(lse == 0.25))
    binding.verify_attn_mla_device_plan(q, dc.kv_pool, dc.kv_indptr, kvi, dc.qo_indptr, B, maxq, maxkv, out, lse, ws,
                                        dc.sm_scale)
    assert binding.verify_attn_mla_check(ws) == binding.VMLA_ERR_INDEX
