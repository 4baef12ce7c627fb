"""A prepared call (arguments checked and marshalled once) gives the plain call's result bit for bit,
also after the contents of its input buffers change between calls."""
import numpy as np
import pytest

from speculative_decoding_mla_gb300 import synth

pytestmark = pytest.mark.gpu


def test_prepared_verify_equals_plain_call_bitwise():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding, device
    case = synth.make_case("prepared", [3000, 500], [16, 5], num_heads=64, pool_slots=3700, seed=51)
    dc = device.to_device(case)
    ref_o, ref_l, ws = device.run(dc, kernel="tc")
    out, lse = device.alloc_outputs(dc)
    call = binding.prepare_verify_attn_mla(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr,
                                           dc.kv_indptr_host, dc.qo_indptr_host, out, lse, ws, dc.sm_scale)
    call()
    torch.cuda.synchronize()
    assert binding.verify_attn_mla_check(ws) == 0
    assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(lse, ref_l)
    # new query contents in the same buffer: the prepared call reads them
    other = synth.make_case("prepared2", [3000, 500], [16, 5], num_heads=64, pool_slots=3700, seed=52)
    dc.q.copy_(torch.from_numpy(other.q.view(np.int16)).view(torch.bfloat16).to(dc.q.device))
    call()
    o2, l2, _ = device.run(dc, kernel="tc")
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), o2.view(torch.int16)) and torch.equal(lse, l2)
    assert not torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
