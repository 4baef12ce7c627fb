"""GPU tests of persistent KV defragmentation and the verify call on pool
runs: defragment a case's scattered rows into runs (in a pool whose other
slots hold NaN patterns), then the runs path equals the per-call-gather path
bit for bit and matches the oracle; runs or slots outside their pools are
reported."""
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


def _bases(case, gap=128):
    n = np.diff(case.kv_indptr).astype(np.int64)
    padded = (n + 127) // 128 * 128 + gap
    base = np.zeros(case.batch, np.int64)
    base[1:] = np.cumsum(padded)[:-1]
    return (base + gap).astype(np.int32), int(base[-1] + padded[-1] + gap) if case.batch else gap


def run_runs(case, splits=0, gap=128):
    torch, binding, device = _mods()
    dc = device.to_device(case)
    base, slots = _bases(case, gap)
    dst = torch.full((slots, 576), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)  # 0xFFFF: NaN
    base_d = torch.from_numpy(base).cuda()
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.verify_attn_mla_defrag(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, dst, base_d, st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    out, lse = device.alloc_outputs(dc)
    ws = torch.empty(max(256, binding.verify_attn_mla_runs_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host,
                                                                           dc.num_heads, splits)),
                     dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_runs(dc.q, dst, dc.kv_indptr, base_d, dc.qo_indptr, dc.kv_indptr_host, dc.qo_indptr_host,
                                 out, lse, ws, dc.sm_scale, parent=dc.parent, splits=splits)
    status = binding.verify_attn_mla_check(ws)
    torch.cuda.synchronize()
    return device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), status


@pytest.mark.parametrize("name", ["one_seq", "ragged", "tree", "heads_odd", "decode_q1"])
def test_runs_equal_gather_path_bitwise(name):
    case = small(name, seed=510)
    o1, l1, s1 = run_full(case, "tc")
    o2, l2, s2 = run_runs(case)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_runs_forced_splits_bitwise():
    case = small("ragged", seed=511)
    o1, l1, _ = run_full(case, "tc", splits=5)
    o2, l2, st = run_runs(case, splits=5, gap=0)
    assert st == 0 and np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_runs_contiguous_1k_against_oracle():
    case = synth.workload("contiguous_1k")
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_runs(case)
    assert st == 0
    compare(o, l, ref_o, ref_l, "runs / contiguous_1k")


def test_runs_and_slots_outside_their_pools_are_reported():
    torch, binding, device = _mods()
    case = small("ragged", seed=512)
    dc = device.to_device(case)
    base, slots = _bases(case)
    dst = torch.zeros((slots, 576), dtype=torch.bfloat16, device="cuda")
    # a source slot past the pool
    bad_idx = dc.kv_indices.clone()
    bad_idx[3] = case.pool_slots + 9
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.verify_attn_mla_defrag(dc.kv_pool, dc.kv_indptr, bad_idx, dc.kv_indptr_host, dst,
                                   torch.from_numpy(base).cuda(), st)
    torch.cuda.synchronize()
    assert int(st[0]) == binding.VMLA_ERR_INDEX and int(st[1]) == 3
    # a run that ends past the destination
    far = base.copy()
    far[1] = slots - 5
    st.zero_()
    binding.verify_attn_mla_defrag(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, dst,
                                   torch.from_numpy(far).cuda(), st)
    torch.cuda.synchronize()
    assert int(st[0]) == binding.VMLA_ERR_INDEX and int(st[1]) == 1
    # the verify call on such a run reports it too
    out, lse = device.alloc_outputs(dc)
    ws = torch.empty(binding.verify_attn_mla_runs_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host,
                                                                 dc.num_heads), dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_runs(dc.q, dst, dc.kv_indptr, torch.from_numpy(far).cuda(), dc.qo_indptr,
                                 dc.kv_indptr_host, dc.qo_indptr_host, out, lse, ws, dc.sm_scale)
    assert binding.verify_attn_mla_check(ws) == binding.VMLA_ERR_INDEX


@pytest.mark.slow
def test_runs_long_185k_sampled_rows():
    """The runs path on the full 185,000-token workload (as the bench times it): bit-equal to the
    per-call gather path, and sampled rows against the oracle."""
    from tests.test_gpu_parity import full_case, oracle_rows, sample_rows
    case = full_case("long_185k")
    o1, l1, s1 = run_full(case, "tc")
    o2, l2, s2 = run_runs(case)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    rows = sample_rows(case)
    ref_o, ref_l = oracle_rows(case, rows, "long_185k/sampled")
    compare(o2.reshape(-1, o2.shape[-1])[rows], l2.reshape(-1)[rows], ref_o, ref_l, "runs / long_185k")


def test_defrag_append_equals_full_defrag():
    """A decode step's append: the runs hold an earlier state (each sequence g_b rows shorter); the append
    copies only rows j >= first_row[b] = N_b - g_b of the new state.  The run regions then equal a full
    defragmentation of the new state bit for bit, and the runs call on them equals the gather path; a
    first_row past N_b is reported."""
    torch, binding, device = _mods()
    case = small("ragged", seed=515)
    dc = device.to_device(case)
    n = np.diff(case.kv_indptr).astype(np.int64)
    rng = np.random.default_rng(516)
    grow = np.array([int(rng.integers(1, k + 1)) if k > 0 else 0 for k in n], np.int64)
    old_n = n - grow
    old_indptr = np.zeros(case.batch + 1, np.int32)
    old_indptr[1:] = np.cumsum(old_n)
    ind = dc.kv_indices.cpu().numpy()
    old_ind = np.concatenate([ind[case.kv_indptr[b]:case.kv_indptr[b] + old_n[b]] for b in range(case.batch)])
    base, slots = _bases(case)
    base_d = torch.from_numpy(base).cuda()

    def nan_pool():
        return torch.full((slots, 576), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)

    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    a = nan_pool()
    binding.verify_attn_mla_defrag(dc.kv_pool, torch.from_numpy(old_indptr).cuda(),
                                   torch.from_numpy(old_ind.astype(np.int32)).cuda(), old_indptr, a, base_d, st)
    first = torch.from_numpy((n - grow).astype(np.int32)).cuda()
    binding.verify_attn_mla_defrag_append(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, a, base_d,
                                          first, st)
    # the same append with the launch bounded by the largest number of new rows
    a2 = nan_pool()
    binding.verify_attn_mla_defrag(dc.kv_pool, torch.from_numpy(old_indptr).cuda(),
                                   torch.from_numpy(old_ind.astype(np.int32)).cuda(), old_indptr, a2, base_d, st)
    binding.verify_attn_mla_defrag_append(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, a2, base_d,
                                          first, st, max_new_rows=int(grow.max()))
    b_pool = nan_pool()
    binding.verify_attn_mla_defrag(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, b_pool, base_d, st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    av = a.view(torch.int16).cpu().numpy()
    a2v = a2.view(torch.int16).cpu().numpy()
    bv = b_pool.view(torch.int16).cpu().numpy()
    for b in range(case.batch):
        lo, hi = int(base[b]), int(base[b]) + int((n[b] + 127) // 128 * 128)
        assert np.array_equal(av[lo:hi], bv[lo:hi]), b
        assert np.array_equal(a2v[lo:hi], bv[lo:hi]), b
    # the runs call on the appended runs equals the gather path
    out, lse = device.alloc_outputs(dc)
    ws = torch.empty(max(256, binding.verify_attn_mla_runs_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host,
                                                                           dc.num_heads, 0)),
                     dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_runs(dc.q, a, dc.kv_indptr, base_d, dc.qo_indptr, dc.kv_indptr_host, dc.qo_indptr_host,
                                 out, lse, ws, dc.sm_scale)
    assert binding.verify_attn_mla_check(ws) == 0
    o1, l1, s1 = run_full(case, "tc")
    assert s1 == 0
    assert np.array_equal(device.bf16_to_f64(out), o1) and np.array_equal(lse.cpu().numpy().astype(np.float64), l1)
    # a first row past a sequence's length is reported, and that sequence is left alone
    bad = first.clone()
    bad[1] = int(n[1]) + 1
    st.zero_()
    binding.verify_attn_mla_defrag_append(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, a, base_d,
                                          bad, st)
    torch.cuda.synchronize()
    assert int(st[0]) == binding.VMLA_ERR_INDEX and int(st[1]) == 1
    # a sequence with more new rows than the stated bound is reported and left alone
    big = int(np.argmax(grow))
    if grow[big] > 1:
        st.zero_()
        before = a.view(torch.int16).clone()
        binding.verify_attn_mla_defrag_append(dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.kv_indptr_host, a,
                                              base_d, first, st, max_new_rows=int(grow[big]) - 1)
        torch.cuda.synchronize()
        assert int(st[0]) == binding.VMLA_ERR_INDEX
        assert torch.equal(a.view(torch.int16), before)  # the rows were already there: nothing changed
