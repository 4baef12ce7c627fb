"""GPU parity of the merge kernel's three row splits.  A merge row takes four, two or one warps,
chosen at launch from the plan's merge rows and largest piece count (the fewest rounds of the row's
loads times waves of resident warps, ties to more warps per row).  Each case below is built so that
the rule picks one split (checked against a restatement of the rule), and its merged rows are
compared with the oracle on sampled rows."""
import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth
from tests.test_gpu_parity import compare, run_full, sample_rows

pytestmark = pytest.mark.gpu


def _mods():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding
    return torch, binding


def warps_per_row(rows, pieces, sms):
    """The launch rule, restated: 64 resident warps per SM; a lane keeps twelve 16-byte loads in
    flight, so a row of 4 / w float4 columns per lane loads 12 w / 4 pieces per round."""
    resident = sms * 64
    best, best_cost = 4, None
    for w in (4, 2, 1):
        batch = 12 // (4 // w)
        cost = max(1, -(-pieces // batch)) * -(-(rows * w) // resident)
        if best_cost is None or cost < best_cost:
            best, best_cost = w, cost
    return best


# name: (prefixes, drafts, heads, forced pieces, expected warps per row)
CASES = {
    "four_warps_two_rounds": ([2032, 4080], 16, 16, 16, 4),  # 512 rows of 16 pieces
    "two_warps": ([300, 310, 320, 330], 16, 64, 3, 2),  # 4096 rows of 3 pieces
    "one_warp": ([300, 260, 290, 330, 310, 280, 270, 320], 16, 64, 2, 1),  # 8192 rows of 2 pieces
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_merge_split_against_oracle(name):
    torch, binding = _mods()
    prefixes, drafts, heads, splits, want = CASES[name]
    case = synth.make_case(f"merge_{name}", prefixes, drafts, num_heads=heads,
                           pool_slots=sum(prefixes) + drafts * len(prefixes) + 77, seed=930 + len(name))
    info, per = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_TC, case.qo_indptr, case.kv_indptr, heads, splits)
    assert np.all(per == splits) and info.merge_rows == case.q.shape[0] * heads
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert warps_per_row(info.merge_rows, info.max_splits, sms) == want
    o, l, st = run_full(case, "tc", splits=splits)
    assert st == 0
    rows = sample_rows(case, n=300, seed=11)
    ref_o, ref_l = oracle.verify_rows(case, rows)
    compare(o.reshape(-1, o.shape[-1])[rows], l.reshape(-1)[rows], ref_o, ref_l, f"merge/{name}")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
