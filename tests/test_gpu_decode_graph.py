"""GPU tests of the capture-safe decode step on pool runs: the device-planned call
on runs (verify_attn_mla_runs_device_plan) equals the host-planned one bit for
bit, and a decode loop captured once as a CUDA graph -- append each step's new
rows to the runs (verify_attn_mla_defrag_append with a bound), then verify on
the runs with the plan made on the device -- replays over growing sequences and
matches the oracle row by row at every step."""
import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth
from tests.test_gpu_parity import compare, small
from tests.test_gpu_runs import _bases, run_runs

pytestmark = pytest.mark.gpu


def _mods():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding, device
    return torch, binding, device


def run_runs_dplan(case, splits=0, slack_q=0, slack_kv=0):
    """The device-planned call on runs of a defragmented copy of the case's rows."""
    torch, binding, device = _mods()
    dc = device.to_device(case)
    base, slots = _bases(case)
    dst = torch.full((slots, 576), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    base_d = torch.from_numpy(base).cuda()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.verify_attn_mla_defrag(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, dst, base_d, st)
    T, H = dc.total_q, dc.num_heads
    maxq, maxkv = T + slack_q, int(case.kv_indptr[-1]) + slack_kv
    q = torch.zeros((max(maxq, 1), H, 576), dtype=torch.bfloat16, device="cuda")
    q[:T] = dc.q
    out = torch.full((max(maxq, 1), H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((max(maxq, 1), H), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.verify_attn_mla_runs_device_plan_workspace_size(case.batch, H, maxq, maxkv, splits),
                     dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_runs_device_plan(q, dst, dc.kv_indptr, base_d, dc.qo_indptr, case.batch, maxq, maxkv,
                                             out, lse, ws, dc.sm_scale, parent=dc.parent, splits=splits)
    status = binding.verify_attn_mla_check(ws)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    return device.bf16_to_f64(out[:T]), lse[:T].cpu().numpy().astype(np.float64), status


@pytest.mark.parametrize("name", ["one_seq", "ragged", "tree", "decode_q1"])
def test_runs_device_plan_equals_host_plan_bitwise(name):
    _, binding, _ = _mods()
    case = small(name, seed=810)
    o1, l1, s1 = run_runs(case)
    o2, l2, s2 = run_runs_dplan(case, slack_q=2, slack_kv=400)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and with the lane plan forced on both
    o3, l3, s3 = run_runs(case, splits=binding.VMLA_SPLITS_LANES)
    o4, l4, s4 = run_runs_dplan(case, splits=binding.VMLA_SPLITS_LANES)
    assert s3 == 0 and s4 == 0
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


def test_runs_device_plan_reports_a_run_outside_the_pool():
    torch, binding, device = _mods()
    case = small("ragged", seed=811)
    dc = device.to_device(case)
    base, slots = _bases(case)
    dst = torch.zeros((slots, 576), dtype=torch.bfloat16, device="cuda")
    far = base.copy()
    far[-1] = slots  # the last sequence's run starts past the pool
    T, H = dc.total_q, dc.num_heads
    out, lse = device.alloc_outputs(dc)
    ws = torch.empty(binding.verify_attn_mla_runs_device_plan_workspace_size(case.batch, H, T, int(case.kv_indptr[-1])),
                     dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_runs_device_plan(dc.q, dst, dc.kv_indptr, torch.from_numpy(far).cuda(), dc.qo_indptr,
                                             case.batch, T, int(case.kv_indptr[-1]), out, lse, ws, dc.sm_scale)
    assert binding.verify_attn_mla_check(ws) == binding.VMLA_ERR_INDEX


def test_captured_decode_loop_on_runs_matches_the_oracle():
    """Three sequences, four drafts per step, three steps: the graph (append + verify on runs with the
    plan made on the device) is captured once at the first step's lengths and replayed with the
    indices, first rows and queries of each later step written into its buffers."""
    torch, binding, device = _mods()
    prefixes, Q, H, steps = [700, 1500, 300], 4, 16, 3
    B = len(prefixes)
    final = synth.make_case("decode_loop", [p + (steps - 1) * Q for p in prefixes], Q, num_heads=H,
                            pool_slots=sum(prefixes) + steps * B * Q + 50, seed=820)
    lists = [final.kv_indices[final.kv_indptr[b]:final.kv_indptr[b + 1]] for b in range(B)]

    def step_case(s):
        n = [p + (s + 1) * Q for p in prefixes]
        kvp = np.zeros(B + 1, np.int32)
        kvp[1:] = np.cumsum(n)
        q = synth.bf16_normals(900 + s, synth.TAG_Q, B * Q * H * 576, 1.0).reshape(B * Q, H, 576)
        return synth.Case(name=f"decode_step{s}", q=q, kv_pool=final.kv_pool, kv_indptr=kvp,
                          kv_indices=np.concatenate([lists[b][:n[b]] for b in range(B)]).astype(np.int32),
                          qo_indptr=(np.arange(B + 1) * Q).astype(np.int32), sm_scale=final.sm_scale)

    cases = [step_case(s) for s in range(steps)]
    cap_kv = int(final.kv_indptr[-1])
    pool = device.to_device(final).kv_pool
    # runs sized for the final lengths, with gaps; the prefixes are defragmented before the loop
    padded = (np.array([len(x) for x in lists]) + 127) // 128 * 128 + 128
    base = np.concatenate([[128], 128 + np.cumsum(padded)[:-1]]).astype(np.int32)
    dst = torch.full((int(base[-1] + padded[-1]), 576), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    base_d = torch.from_numpy(base).cuda()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    pre_kvp = np.concatenate([[0], np.cumsum(prefixes)]).astype(np.int32)
    pre_idx = np.concatenate([lists[b][:prefixes[b]] for b in range(B)]).astype(np.int32)
    binding.verify_attn_mla_defrag(pool, torch.from_numpy(pre_kvp).cuda(), torch.from_numpy(pre_idx).cuda(), pre_kvp,
                                   dst, base_d, st)
    # the buffers the graph reads (written before each replay)
    kvp_d = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    kvi_d = torch.zeros(cap_kv, dtype=torch.int32, device="cuda")
    qop_d = torch.from_numpy(cases[0].qo_indptr).cuda()
    first_d = torch.zeros(B, dtype=torch.int32, device="cuda")
    q_d = torch.zeros((B * Q, H, 576), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((B * Q, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B * Q, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.verify_attn_mla_runs_device_plan_workspace_size(B, H, B * Q, cap_kv),
                     dtype=torch.uint8, device="cuda")

    def load(c):
        kvp_d.copy_(torch.from_numpy(c.kv_indptr))
        kvi_d[:len(c.kv_indices)].copy_(torch.from_numpy(c.kv_indices))
        first_d.copy_(torch.from_numpy((np.diff(c.kv_indptr) - Q).astype(np.int32)))
        q_d.copy_(device.to_device(c).q)
        torch.cuda.synchronize()

    load(cases[0])
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        binding.verify_attn_mla_defrag_append(pool, kvp_d, kvi_d, cases[0].kv_indptr, dst, base_d, first_d, st,
                                              max_new_rows=Q)
        binding.verify_attn_mla_runs_device_plan(q_d, dst, kvp_d, base_d, qop_d, B, B * Q, cap_kv, out, lse, ws,
                                                 final.sm_scale)
    for s, c in enumerate(cases):
        load(c)
        graph.replay()
        torch.cuda.synchronize()
        assert int(st[0]) == 0 and binding.verify_attn_mla_check(ws) == 0, s
        ref_o, ref_l = oracle.verify(c)
        compare(device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_o, ref_l, f"decode step {s}")
