"""The allocation-free entry point (collected last on purpose).

verify_attn_mla_simt_static serves callers that cannot allocate device memory
when they call in -- an engine whose free HBM already belongs to its KV cache,
an allocator that must not be re-entered from a callback, a plugin host that
allows cudaMalloc only during its own set-up.  It runs the CUDA-core path on
the library's fixed scratch array.  Both entry points run the same kernels on
the same plan, so their outputs must agree bit for bit; three calls in a row
with different shapes, masks and forced split counts check that nothing one
call leaves in the shared array (ancestor masks, partial rows) reaches the
next.
"""
import numpy as np
import pytest

from speculative_decoding_mla_gb300 import synth

pytestmark = pytest.mark.gpu


def _mods():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding, device
    return torch, binding, device


def _both(case, splits):
    torch, binding, device = _mods()
    dc = device.to_device(case)
    ref_out, ref_lse, ws = device.run(dc, kernel="simt", splits=splits)
    assert binding.verify_attn_mla_check(ws) == 0
    out, lse = device.alloc_outputs(dc)
    out.fill_(7.0)
    lse.fill_(7.0)
    binding.verify_attn_mla_simt_static(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                        dc.kv_indptr_host, dc.qo_indptr_host, out, lse, dc.sm_scale,
                                        draft_mask=dc.draft_mask, parent=dc.parent, splits=splits)
    assert binding.verify_attn_mla_simt_static_check() == 0
    torch.cuda.synchronize()
    return (out.view(torch.int16).cpu().numpy(), lse.cpu().numpy(), ref_out.view(torch.int16).cpu().numpy(),
            ref_lse.cpu().numpy())


def test_static_scratch_matches_workspace_path_bitwise_on_three_calls():
    # causal, then a tree (its ancestor masks and partials follow the causal call's), then a
    # different tree with other lengths and split count over what the first tree left behind
    calls = [
        (synth.make_case("static_causal", [2500, 0, 700], [16, 3, 1], num_heads=64, pool_slots=3300, seed=42), 5),
        (synth.make_case("static_tree", [900, 33], [64, 7], num_heads=16, pool_slots=1100, tree_depth=8, seed=41), 3),
        (synth.make_case("static_tree2", [1500], [40], num_heads=32, pool_slots=1600, tree_depth=4, seed=44), 7),
    ]
    for case, splits in calls:
        o, l, ro, rl = _both(case, splits)
        assert np.array_equal(o, ro), case.name
        assert np.array_equal(l.view(np.uint32), rl.view(np.uint32)), case.name


def test_static_scratch_reports_a_bad_slot():
    torch, binding, device = _mods()
    case = synth.make_case("static_bad", [300], [4], num_heads=8, pool_slots=400, seed=45)
    dc = device.to_device(case)
    dc.kv_indices[17] = 400  # one slot outside the pool
    out, lse = device.alloc_outputs(dc)
    binding.verify_attn_mla_simt_static(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                        dc.kv_indptr_host, dc.qo_indptr_host, out, lse, dc.sm_scale)
    assert binding.verify_attn_mla_simt_static_check() == binding.VMLA_ERR_INDEX
    # the next clean call starts from a cleared status word
    dc.kv_indices[17] = 0
    binding.verify_attn_mla_simt_static(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                        dc.kv_indptr_host, dc.qo_indptr_host, out, lse, dc.sm_scale)
    assert binding.verify_attn_mla_simt_static_check() == 0


def test_static_scratch_rejects_plans_beyond_its_size():
    torch, binding, device = _mods()
    # 64 drafts x 128 heads = 8192 rows split 64 ways needs 8192 * 64 * 2 KB of partials (> 32 MiB)
    case = synth.make_case("too_big", [70000], [64], num_heads=128, pool_slots=70100, seed=43)
    info, _ = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_SIMT, case.qo_indptr, case.kv_indptr, 128, 64)
    assert info.workspace_bytes > binding.STATIC_SCRATCH_BYTES
    dc = device.to_device(case)
    out, lse = device.alloc_outputs(dc)
    with pytest.raises(binding.VmlaError) as e:
        binding.verify_attn_mla_simt_static(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                            dc.kv_indptr_host, dc.qo_indptr_host, out, lse, dc.sm_scale, splits=64)
    assert e.value.status == binding.VMLA_ERR_WORKSPACE
