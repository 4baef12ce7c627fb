"""The allocation-free entry point (collected last on purpose).

verify_attn_mla_simt_static serves callers that cannot allocate device memory
when they call in; it runs the CUDA-core path on the library's fixed scratch
array.  Its output must match verify_attn_mla_simt (which takes a workspace) on
two calls in a row, with different shapes and masks, so that anything the
first call leaves in the shared array cannot leak into the second.
"""
import numpy as np
import pytest

from speculative_decoding_mla_gb300 import synth

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


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
    torch.cuda.synchronize()
    return (device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64),
            device.bf16_to_f64(ref_out), ref_lse.cpu().numpy().astype(np.float64))


def test_static_scratch_matches_workspace_path_on_two_calls():
    first = synth.make_case("static_tree", [900, 33], [64, 7], num_heads=16, pool_slots=1100, tree_depth=8, seed=41)
    second = synth.make_case("static_causal", [2500, 0, 700], [16, 3, 1], num_heads=64, pool_slots=3300, seed=42)
    for case, splits in ((first, 3), (second, 0)):
        o, l, ro, rl = _both(case, splits)
        assert np.max(np.abs(o - ro)) <= OUT_TOL
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(l), fin)
        assert np.max(np.abs(l[fin] - rl[fin])) <= LSE_TOL


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
