"""GPU tests of the e4m3 (fp8) latent pool: the gather dequantizes each row as
the oracle defines it, so the fp8 call equals the bf16 call on the oracle's
dequantized pool bit for bit, and matches the oracle within the tolerance."""
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


def quantize(case):
    """(e4m3 codes [S, 576] uint8, scale, the case with the oracle's dequantized bf16 pool)."""
    import torch
    vals = synth.bf16_bits_to_f64(case.kv_pool).astype(np.float32)
    scale = float(np.abs(vals).max() / 400.0)  # not a power of two: the float32 product rounds
    codes = (torch.from_numpy(vals) / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    deq = oracle.dequantize_e4m3(codes, scale).reshape(case.kv_pool.shape)
    case2 = synth.Case(name=case.name + "_fp8", q=case.q, kv_pool=deq, kv_indptr=case.kv_indptr,
                       kv_indices=case.kv_indices, qo_indptr=case.qo_indptr, parent=case.parent,
                       sm_scale=case.sm_scale)
    return codes, scale, case2


def run_fp8(case, codes, scale, splits=0):
    torch, binding, device = _mods()
    dc = device.to_device(case)
    pool = torch.from_numpy(codes).cuda()
    out, lse = device.alloc_outputs(dc)
    ws = device.alloc_workspace(dc, splits)
    binding.verify_attn_mla_fp8(dc.q, pool, scale, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, dc.kv_indptr_host,
                                dc.qo_indptr_host, out, lse, ws, dc.sm_scale, parent=dc.parent, splits=splits)
    st = binding.verify_attn_mla_check(ws)
    torch.cuda.synchronize()
    return device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), st


@pytest.mark.parametrize("name", ["one_seq", "ragged", "tree", "decode_q1"])
def test_fp8_equals_bf16_on_the_dequantized_pool(name):
    case = small(name, seed=610)
    codes, scale, deq_case = quantize(case)
    o1, l1, s1 = run_full(deq_case, "tc")
    o2, l2, s2 = run_fp8(case, codes, scale)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_contiguous_1k_against_oracle():
    case = synth.workload("contiguous_1k")
    codes, scale, deq_case = quantize(case)
    ref_o, ref_l = oracle.verify(deq_case)
    o, l, st = run_fp8(case, codes, scale, splits=3)
    assert st == 0
    compare(o, l, ref_o, ref_l, "fp8 / contiguous_1k")


def test_fp8_bad_slot_is_reported():
    _, binding, _ = _mods()
    case = small("one_seq", seed=611)
    codes, scale, _ = quantize(case)
    case.kv_indices = case.kv_indices.copy()
    case.kv_indices[5] = case.pool_slots + 3
    _, l, st = run_fp8(case, codes, scale)
    assert st == binding.VMLA_ERR_INDEX and np.all(np.isfinite(l))


@pytest.mark.slow
def test_fp8_long_185k_sampled_rows():
    """The e4m3 pool path on the full 185,000-token workload: sampled rows against the oracle on the
    dequantized pool, and bit-equal to the bf16 call on that pool."""
    from tests.test_gpu_parity import full_case, run_full, sample_rows
    case = full_case("long_185k")
    codes, scale, case2 = quantize(case)
    o, l, st = run_fp8(case, codes, scale)
    assert st == 0
    o2, l2, s2 = run_full(case2, "tc")
    assert s2 == 0
    assert np.array_equal(o, o2) and np.array_equal(l, l2)
    rows = sample_rows(case)
    ref_o, ref_l = oracle.verify_rows(case2, rows)
    compare(o.reshape(-1, o.shape[-1])[rows], l.reshape(-1)[rows], ref_o, ref_l, "fp8 / long_185k")
