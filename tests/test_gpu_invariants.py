"""GPU checks of properties, of the merge and mask kernels on their own, of the
host-buffer entry point, and of the faults kernels report (bad slot index,
malformed parents) through the workspace status word."""
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


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_permuted_pool_bitwise(kernel):
    case = small("ragged", seed=300)
    o1, l1, _ = run_full(case, kernel)
    pi = synth.permutation(7, synth.TAG_AUX, case.pool_slots)
    pool2 = np.empty_like(case.kv_pool)
    pool2[pi] = case.kv_pool
    case2 = synth.Case(name="perm", q=case.q, kv_pool=pool2, kv_indptr=case.kv_indptr,
                       kv_indices=pi[case.kv_indices].astype(np.int32), qo_indptr=case.qo_indptr,
                       sm_scale=case.sm_scale)
    o2, l2, _ = run_full(case2, kernel)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_parent_chain_equals_causal_bitwise(kernel):
    case = small("ragged", seed=301)
    o1, l1, _ = run_full(case, kernel)
    chain = []
    for b in range(case.batch):
        n = int(case.qo_indptr[b + 1] - case.qo_indptr[b])
        chain += list(range(-1, n - 1))
    case.parent = np.array(chain, np.int32)
    o2, l2, _ = run_full(case, kernel)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_zero_queries_give_mean():
    case = small("one_seq", seed=302)
    case.q[:] = 0
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, "tc")
    compare(o, l, ref_o, ref_l, "q = 0")


def test_merge_kernel_alone():
    torch, binding, device = _mods()
    rng = np.random.default_rng(3)
    S, R = 7, 300
    o_parts = rng.normal(size=(S, R, 512)).astype(np.float32)
    lse_parts = rng.normal(scale=3.0, size=(S, R)).astype(np.float32)
    lse_parts[2, :50] = -np.inf
    lse_parts[:, 7] = -np.inf  # a row with every part empty
    ref_o, ref_l = oracle.merge(o_parts.astype(np.float64), lse_parts.astype(np.float64))
    o_parts[2, :50] = np.nan  # an empty piece's partial row carries no weight, whatever it holds
    out = torch.empty((R, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(R, dtype=torch.float32, device="cuda")
    binding.verify_attn_mla_merge(torch.from_numpy(o_parts).cuda(), torch.from_numpy(lse_parts).cuda(), out, lse)
    torch.cuda.synchronize()
    compare(device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_o, ref_l, "merge")


def test_tree_mask_kernel_alone():
    torch, binding, device = _mods()
    parents = np.concatenate([synth.tree_parents(9, n, 8, s) for s, n in enumerate([64, 1, 17, 40])])
    qo = np.array([0, 64, 65, 82, 122], np.int32)
    ref = oracle.tree_masks(parents, qo)
    out = torch.empty(len(parents), dtype=torch.int64, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.verify_attn_mla_tree_mask(torch.from_numpy(parents).cuda(), torch.from_numpy(qo).cuda(), out, st)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint64), ref)
    assert int(st[0]) == 0


def test_bad_parent_is_reported():
    torch, binding, device = _mods()
    case = small("tree", seed=303)
    case.parent = case.parent.copy()
    case.parent[5] = 9  # a parent after its child
    o, l, st = run_full(case, "tc")
    assert st == binding.VMLA_ERR_PARENT


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_bad_slot_index_is_reported(kernel):
    torch, binding, device = _mods()
    case = small("one_seq", seed=304)
    case.kv_indices = case.kv_indices.copy()
    case.kv_indices[17] = case.pool_slots + 5
    o, l, st = run_full(case, kernel)
    assert st == binding.VMLA_ERR_INDEX
    assert np.all(np.isfinite(l))


def test_host_entry_point_matches_device_path():
    torch, binding, device = _mods()
    case = small("tree", seed=305)
    o1, l1, _ = run_full(case, "tc")
    kv = device.to_device(case).kv_pool
    T, H = case.q.shape[0], case.num_heads
    q_h = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    out_h = torch.empty((T, H, 512), dtype=torch.int16).pin_memory()
    lse_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    kvi_h = torch.from_numpy(case.kv_indices).pin_memory()
    par_h = torch.from_numpy(case.parent).pin_memory()
    n = binding.verify_attn_mla_host_buffer_size(case.qo_indptr, case.kv_indptr, H, has_parent=True)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla_host(q_h, kv, case.kv_indptr, kvi_h, case.qo_indptr, out_h, lse_h, buf, case.sm_scale,
                                 parent_host=par_h)
    o2 = synth.bf16_bits_to_f64(out_h.numpy().view(np.uint16))
    assert np.array_equal(o1, o2) and np.array_equal(l1, lse_h.numpy().astype(np.float64))


def test_host_entry_point_indices_pageable_pinned_and_offset():
    """The host-buffer call reads page-locked indices in place (through their mapped device address)
    and copies other host memory first: pageable indices, pinned indices, and pinned indices that
    start inside their allocation all give the device call's bits, with an explicit draft mask."""
    torch, binding, device = _mods()
    case = small("ragged", seed=312)
    T, H = case.q.shape[0], case.num_heads
    rng = np.random.default_rng(5)
    mask = np.zeros(T, dtype=np.uint64)
    for b in range(case.batch):
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        for i in range(q1 - q0):
            bits = int(rng.integers(0, 1 << max(i, 1))) & ((1 << i) - 1)
            mask[q0 + i] = np.uint64(bits | (1 << i))
    o1, l1, st = run_full(case, "tc", draft_mask=mask)
    assert st == 0
    kv = device.to_device(case).kv_pool
    q_h = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    m_h = torch.from_numpy(mask.view(np.int64)).pin_memory()
    n = binding.verify_attn_mla_host_buffer_size(case.qo_indptr, case.kv_indptr, H, has_mask=True)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    N = len(case.kv_indices)
    pinned_big = torch.zeros(N + 37, dtype=torch.int32).pin_memory()
    pinned_big[37:] = torch.from_numpy(case.kv_indices)
    for what, kvi_h in [("pageable", torch.from_numpy(case.kv_indices.copy())),
                        ("pinned", torch.from_numpy(case.kv_indices).pin_memory()),
                        ("pinned, offset", pinned_big[37:])]:
        assert kvi_h.is_pinned() == (what != "pageable")
        out_h = torch.full((T, H, 512), -1, dtype=torch.int16).pin_memory()
        lse_h = torch.full((T, H), float("nan"), dtype=torch.float32).pin_memory()
        binding.verify_attn_mla_host(q_h, kv, case.kv_indptr, kvi_h, case.qo_indptr, out_h, lse_h, buf,
                                     case.sm_scale, draft_mask_host=m_h)
        o2 = synth.bf16_bits_to_f64(out_h.numpy().view(np.uint16))
        assert np.array_equal(o1, o2) and np.array_equal(l1, lse_h.numpy().astype(np.float64)), what


def test_host_entry_point_reports_a_bad_slot():
    """The host-buffer call returns the device status word (read back with its results): a slot
    outside the pool gives VMLA_ERR_INDEX, and the next good call on the same buffers returns 0."""
    torch, binding, device = _mods()
    case = small("ragged", seed=308)
    kv = device.to_device(case).kv_pool
    T, H = case.q.shape[0], case.num_heads
    q_h = torch.from_numpy(case.q.view(np.int16)).pin_memory()
    out_h = torch.empty((T, H, 512), dtype=torch.int16).pin_memory()
    lse_h = torch.empty((T, H), dtype=torch.float32).pin_memory()
    bad = case.kv_indices.copy()
    bad[3] = case.pool_slots + 7
    kvi_h = torch.from_numpy(bad).pin_memory()
    n = binding.verify_attn_mla_host_buffer_size(case.qo_indptr, case.kv_indptr, H)
    buf = torch.empty(n, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.VmlaError) as err:
        binding.verify_attn_mla_host(q_h, kv, case.kv_indptr, kvi_h, case.qo_indptr, out_h, lse_h, buf,
                                     case.sm_scale)
    assert err.value.status == binding.VMLA_ERR_INDEX
    kvi_h.copy_(torch.from_numpy(case.kv_indices))
    binding.verify_attn_mla_host(q_h, kv, case.kv_indptr, kvi_h, case.qo_indptr, out_h, lse_h, buf, case.sm_scale)
    o1, l1, _ = run_full(case, "tc")
    o2 = synth.bf16_bits_to_f64(out_h.numpy().view(np.uint16))
    assert np.array_equal(o1, o2) and np.array_equal(l1, lse_h.numpy().astype(np.float64))


def test_empty_batch_and_empty_sequences():
    torch, binding, device = _mods()
    case = synth.make_case("empties", [0, 40, 0], [0, 3, 0], num_heads=8, pool_slots=60, seed=306)
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, "tc")
    assert st == 0
    compare(o, l, ref_o, ref_l, "empties")
    case0 = synth.make_case("none", [], [], num_heads=8, pool_slots=1, seed=307)
    dc = device.to_device(case0)
    out, lse = device.alloc_outputs(dc)
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, dc.kv_indptr_host,
                            dc.qo_indptr_host, out, lse, ws, dc.sm_scale)
    assert binding.verify_attn_mla_check(ws) == 0


def test_small_workspace_is_rejected():
    torch, binding, device = _mods()
    case = small("ragged", seed=308)
    dc = device.to_device(case)
    out, lse = device.alloc_outputs(dc)
    n = binding.verify_attn_mla_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host, dc.num_heads, 7)
    # far below the staged KV rows alone (1152 bytes per key)
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    assert n > 1024
    with pytest.raises(binding.VmlaError) as e:
        binding.verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, dc.kv_indptr_host,
                                dc.qo_indptr_host, out, lse, ws, dc.sm_scale, splits=7)
    assert e.value.status == binding.VMLA_ERR_WORKSPACE


def test_workspace_short_of_the_partials_only_is_rejected_after_the_gather():
    """A workspace that holds the status word, masks and staged rows but not the plan's
    partials: the call queues the gather (planned afterwards, on the host) and then reports
    VMLA_ERR_WORKSPACE; out and lse are untouched, and a call with enough room is correct."""
    torch, binding, device = _mods()
    case = small("ragged", seed=309)
    dc = device.to_device(case)
    T, N = int(case.qo_indptr[-1]), int(case.kv_indptr[-1])
    up = lambda x: (x + 255) // 256 * 256
    n_rows = 256 + up(T * 8) + up(N * 1152)  # status, masks, staged rows
    n_full = binding.verify_attn_mla_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host, dc.num_heads, 7)
    assert n_full > n_rows
    out = torch.full((T, dc.num_heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, dc.num_heads), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(n_rows, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.VmlaError) as e:
        binding.verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, dc.kv_indptr_host,
                                dc.qo_indptr_host, out, lse, ws, dc.sm_scale, splits=7)
    assert e.value.status == binding.VMLA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    ws2 = torch.empty(n_full, dtype=torch.uint8, device="cuda")
    binding.verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, dc.kv_indptr_host,
                            dc.qo_indptr_host, out, lse, ws2, dc.sm_scale, splits=7)
    assert binding.verify_attn_mla_check(ws2) == 0
    ref_o, ref_l = oracle.verify(case)
    compare(device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), ref_o, ref_l, "after a short workspace")


def test_bounded_wait_expiry_reports_timeout_and_context_stays_usable():
    """A signal that never comes (the test flag withholds Q-ready): the kernel's bounded wait
    expires, the status word says VMLA_ERR_TIMEOUT, and the next call works normally."""
    torch, binding, device = _mods()
    case = small("one_seq", seed=320)
    dc = device.to_device(case)
    try:
        binding.verify_attn_mla_test_fault(1, 20_000_000)  # ~10 ms per bounded wait
        _, _, ws = device.run(dc, kernel="tc")
        st = binding.verify_attn_mla_check(ws)  # the outputs of this call are not defined
    finally:
        binding.verify_attn_mla_test_fault(0, 0)
    assert st == binding.VMLA_ERR_TIMEOUT
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, "tc")
    assert st == 0
    compare(o, l, ref_o, ref_l, "after the failure test")
