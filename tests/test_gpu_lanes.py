"""GPU tests of the tensor-core kernel's lane plan: the clusters form lanes of G,
each sequence's G-row-block streams are laid end to end and cut where the
lanes' shares end, and a stream cut into several pieces is combined by the
merge while a stream inside one lane writes its rows directly.  Every row is
compared with the oracle; the device planner's lane plan equals the host
planner's bit for bit, and so does the call on pool runs."""
import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth
from tests.test_gpu_dplan import run_dplan
from tests.test_gpu_parity import compare, full_case, oracle_rows, run_full
from tests.test_gpu_runs import run_runs

pytestmark = pytest.mark.gpu

# (prefixes, drafts, heads, tree depth): lane widths 1 (one row block per sequence), 2, 3 and 4,
# a sequence without drafts between others, trees, and a head count that leaves a ragged row block
LANE_CASES = {
    "g1_decode": ([3000, 500, 9000, 1200, 0, 7000, 2500], [2, 4, 1, 3, 2, 4, 1], 64, None),
    "g1_zero_drafts": ([3000, 4000, 100, 6000], [4, 0, 4, 4], 64, None),
    "g2": ([2000, 500, 5000, 800], [8] * 4, 64, None),
    "g3": ([2000, 700, 4000], [12] * 3, 64, None),
    "g4_ragged": ([900, 3000, 6000, 1500, 200], [16] * 5, 64, None),
    "g4_tree": ([3000, 600, 1200], [64, 64, 64], 16, 8),
    "g1_heads_odd": ([77, 2000, 5000], [5, 2, 7], 12, None),
}
WIDTH = {"g1_decode": 1, "g1_zero_drafts": 1, "g2": 2, "g3": 3, "g4_ragged": 4, "g4_tree": 4, "g1_heads_odd": 1}


def lane_case(name, seed=700):
    pre, drafts, heads, tree = LANE_CASES[name]
    return synth.make_case(name, pre, drafts, num_heads=heads, pool_slots=sum(pre) + sum(drafts) + 57,
                           tree_depth=tree, seed=seed)


def _lanes():
    from speculative_decoding_mla_gb300 import binding
    return binding


def _plan_info(case, splits):
    binding = _lanes()
    info, per = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_TC, case.qo_indptr, case.kv_indptr,
                                             case.num_heads, splits, 144)
    return info, per


@pytest.mark.parametrize("name", sorted(LANE_CASES))
def test_lane_plan_every_row(name):
    """VMLA_SPLITS_LANES on small cases: the lane plan of the expected width, cut into more than one
    piece somewhere (so both the merge and the direct writes run), against the oracle row by row."""
    binding = _lanes()
    case = lane_case(name)
    info, per = _plan_info(case, binding.VMLA_SPLITS_LANES)
    assert info.lane_width == WIDTH[name]
    assert int(np.max(per)) > 1
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, "tc", splits=binding.VMLA_SPLITS_LANES)
    assert st == 0
    compare(o, l, ref_o, ref_l, f"lanes/{name}")


@pytest.mark.parametrize("name", ["g1_decode", "g3", "g4_tree"])
def test_lane_plan_device_planner_bitwise(name):
    """The device planner builds the same lane plan as the host planner: identical results."""
    binding = _lanes()
    case = lane_case(name, seed=701)
    o1, l1, s1 = run_full(case, "tc", splits=binding.VMLA_SPLITS_LANES)
    slack_q = 0 if name == "g4_tree" else 3  # 64-node trees: the query bound is already the most allowed
    o2, l2, s2 = run_dplan(case, splits=binding.VMLA_SPLITS_LANES, slack_q=slack_q, slack_kv=500)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("name", ["g1_zero_drafts", "g4_ragged"])
def test_lane_plan_on_pool_runs_bitwise(name):
    """The call on defragmented pool runs under a lane plan equals the gather path's bit for bit."""
    binding = _lanes()
    case = lane_case(name, seed=702)
    o1, l1, s1 = run_full(case, "tc", splits=binding.VMLA_SPLITS_LANES)
    o2, l2, s2 = run_runs(case, splits=binding.VMLA_SPLITS_LANES)
    assert s1 == 0 and s2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["paged_ragged", "sweep_q1"])
def test_full_size_lane_plan_every_row(name):
    """The planner's own choice on the ragged 4k-32k batch (lanes of four clusters) and on the 32
    lognormal sequences with one draft (lanes of one cluster): every query row against the oracle,
    in the configuration the bench times."""
    binding = _lanes()
    case = full_case(name)
    info, _ = _plan_info(case, 0)
    assert info.lane_width > 0
    rows = np.arange(case.q.shape[0] * case.num_heads, dtype=np.int64)
    ref_o, ref_l = oracle_rows(case, rows, f"{name}/all")
    o, l, st = run_full(case, "tc")
    assert st == 0
    compare(o.reshape(-1, o.shape[-1]), l.reshape(-1), ref_o, ref_l, f"tc/{name} every row")


def test_lane_plan_many_sequences_every_row():
    """VMLA_SPLITS_LANES on 80 short sequences (past the candidate search's 64, so the device
    planner takes its forced path): lanes of one cluster meeting up to five streams, several lanes
    starting inside a stream's fixed charge; every row against the oracle, and the device plan
    bit for bit."""
    binding = _lanes()
    rng = np.random.default_rng(900)
    prefixes = rng.integers(50, 3000, 80).tolist()
    drafts = rng.integers(1, 5, 80).tolist()
    case = synth.make_case("lanes_b80", prefixes, drafts, num_heads=64,
                           pool_slots=sum(prefixes) + sum(drafts) + 99, seed=703)
    info, per = _plan_info(case, binding.VMLA_SPLITS_LANES)
    assert info.lane_width == 1 and int(np.max(per)) > 1
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, "tc", splits=binding.VMLA_SPLITS_LANES)
    assert st == 0
    compare(o, l, ref_o, ref_l, "lanes/b80")
    o2, l2, s2 = run_dplan(case, splits=binding.VMLA_SPLITS_LANES, slack_q=7, slack_kv=300)
    assert s2 == 0
    assert np.array_equal(o, o2) and np.array_equal(l, l2)
