"""GPU parity: the CUDA path against the CPU fp64 oracle on the same seeded inputs.

Tolerances (the target's own): max |out_gpu - out_oracle| <= 1e-2 on the bf16
output and max |lse_gpu - lse_oracle| <= 1e-3 on the fp32 log-sum-exp.
Small cases are compared element by element over every row; the full-size
workloads run in the launch configuration the bench times and are compared
on every row of the 185,000-token workload, every row of one 256-row unit per
sequence of the tree and Q=4 sweep workloads, and sampled rows of all of them,
which the oracle evaluates one by one.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3
KERNELS = ["tc", "simt"]


def _dev():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import device
    return torch, device


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    err_o = float(np.max(np.abs(out_gpu - out_ref))) if out_ref.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), f"{what}: -inf pattern differs"
    err_l = float(np.max(np.abs(lse_gpu[fin] - lse_ref[fin]))) if fin.any() else 0.0
    assert err_o <= OUT_TOL, f"{what}: max out error {err_o}"
    assert err_l <= LSE_TOL, f"{what}: max lse error {err_l}"
    return err_o, err_l


def run_full(case, kernel, splits=0, draft_mask=None):
    torch, device = _dev()
    dc = device.to_device(case, draft_mask=draft_mask)
    out, lse, ws = device.run(dc, kernel=kernel, splits=splits)
    from speculative_decoding_mla_gb300 import binding
    st = binding.verify_attn_mla_check(ws)
    torch.cuda.synchronize()
    return device.bf16_to_f64(out), lse.cpu().numpy().astype(np.float64), st


SMALL = {
    "one_seq": dict(prefixes=[300], drafts=16, heads=64, tree=None),
    "ragged": dict(prefixes=[0, 129, 1000, 7], drafts=[3, 16, 1, 64], heads=8, tree=None),
    "tree": dict(prefixes=[500, 64], drafts=[64, 20], heads=16, tree=8),
    "heads_odd": dict(prefixes=[77, 2000], drafts=[5, 2], heads=12, tree=None),
    "decode_q1": dict(prefixes=[1500] * 5, drafts=1, heads=64, tree=None),
}


def small(name, seed=200):
    s = SMALL[name]
    drafts = s["drafts"]
    nd = sum(drafts) if isinstance(drafts, list) else drafts * len(s["prefixes"])
    return synth.make_case(name, s["prefixes"], drafts, num_heads=s["heads"],
                           pool_slots=sum(s["prefixes"]) + nd + 33, tree_depth=s["tree"], seed=seed)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_every_row(kernel, name):
    case = small(name)
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, kernel)
    assert st == 0
    compare(o, l, ref_o, ref_l, f"{kernel}/{name}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_contiguous_1k_every_row(kernel):
    case = synth.workload("contiguous_1k")
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, kernel)
    assert st == 0
    compare(o, l, ref_o, ref_l, "contiguous_1k")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_forced_splits(kernel, splits):
    case = small("ragged", seed=201)
    ref_o, ref_l = oracle.verify(case)
    o, l, st = run_full(case, kernel, splits=splits)
    assert st == 0
    compare(o, l, ref_o, ref_l, f"splits={splits}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_explicit_mask_and_empty_rows(kernel):
    case = small("ragged", seed=202)
    T = case.q.shape[0]
    rng = np.random.default_rng(5)
    dm = rng.integers(0, 2 ** 63, size=T, dtype=np.int64).astype(np.uint64)
    dm[0] = 0  # first sequence has no prefix: query 0 sees nothing -> out 0, lse -inf
    ref_o, ref_l = oracle.verify(case, draft_mask=dm)
    assert not np.isfinite(ref_l[0]).any()
    o, l, st = run_full(case, kernel, draft_mask=dm)
    assert st == 0
    compare(o, l, ref_o, ref_l, "explicit mask")
    assert np.all(o[0] == 0.0)


def sample_rows(case, n=40, seed=0):
    """Rows spread over every sequence: first/last query and head of each, plus seeded extras."""
    H = case.num_heads
    rows = set()
    for b in range(case.batch):
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        if q1 == q0:
            continue
        rows |= {q0 * H, q0 * H + H - 1, (q1 - 1) * H, q1 * H - 1}
    w = synth.words(seed, synth.TAG_AUX, n)
    total = case.q.shape[0] * H
    rows |= {int(x % np.uint64(total)) for x in w}
    return np.array(sorted(rows), dtype=np.int64)


_FULL = {}


def full_case(name):
    if name not in _FULL:
        _FULL[name] = synth.workload(name)
    return _FULL[name]


@pytest.mark.slow
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", ["paged_ragged", "long_185k", "tree_32k", "sweep_q1", "sweep_q4", "sweep_q16"])
def test_full_size_sampled_rows(kernel, name):
    case = full_case(name)
    o, l, st = run_full(case, kernel)
    assert st == 0
    rows = sample_rows(case)
    ref_o, ref_l = oracle.verify_rows(case, rows)
    H = case.num_heads
    og = o.reshape(-1, o.shape[-1])[rows]
    lg = l.reshape(-1)[rows]
    compare(og, lg, ref_o, ref_l, f"{kernel}/{name}")
    # properties that hold for every row: finite, and each output is a convex
    # combination of latent rows, so it lies inside the pool's value range
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    pool = synth.bf16_bits_to_f64(case.kv_pool[:, :512])
    assert o.max() <= pool.max() + OUT_TOL and o.min() >= pool.min() - OUT_TOL


@pytest.mark.parametrize("kernel", KERNELS)
def test_maximum_heads_and_drafts(kernel):
    """128 heads x 64 drafts (8192 query rows per sequence): the largest row count a sequence can have."""
    case = synth.make_case("max_rows", [300, 1500], 64, num_heads=128, pool_slots=2000, seed=211)
    o, l, st = run_full(case, kernel)
    assert st == 0
    rows = sample_rows(case, n=300, seed=3)
    ref_o, ref_l = oracle.verify_rows(case, rows)
    compare(o.reshape(-1, o.shape[-1])[rows], l.reshape(-1)[rows], ref_o, ref_l, f"{kernel}/max_rows")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))


def test_more_units_than_one_launch_holds():
    """4096 tensor-core work units (16 sequences x 4 row pairs x 64 forced pieces) run as two launches."""
    from speculative_decoding_mla_gb300 import binding
    case = synth.make_case("many_units", [8176] * 16, 16, num_heads=64, pool_slots=16 * 8192 + 50, seed=212)
    info, per = binding.verify_attn_mla_plan(binding.VMLA_KERNEL_TC, case.qo_indptr, case.kv_indptr, 64, 64)
    assert info.num_units == 4096 and np.all(per == 64)
    o, l, st = run_full(case, "tc", splits=64)
    assert st == 0
    rows = sample_rows(case, n=200, seed=4)
    ref_o, ref_l = oracle.verify_rows(case, rows)
    compare(o.reshape(-1, o.shape[-1])[rows], l.reshape(-1)[rows], ref_o, ref_l, "many_units")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))


_ORACLE_ROWS = {}


def oracle_rows(case, rows, key):
    """The oracle's result for `rows` of a full-size case, computed once per test session."""
    if key not in _ORACLE_ROWS:
        _ORACLE_ROWS[key] = oracle.verify_rows(case, rows)
    return _ORACLE_ROWS[key]


def unit_rows(case, rows_per_unit=256):
    """Every row of the first 256-row unit (row block 0) of each sequence."""
    H = case.num_heads
    out = []
    for b in range(case.batch):
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        n = (q1 - q0) * H
        out.append(q0 * H + np.arange(min(n, rows_per_unit), dtype=np.int64))
    return np.concatenate(out)


@pytest.mark.slow
@pytest.mark.parametrize("kernel", KERNELS)
def test_long_185k_every_row(kernel):
    """All 1024 query rows (16 drafts x 64 heads) of the 185,000-token workload, in the bench's launch
    configuration, against the oracle row by row."""
    case = full_case("long_185k")
    rows = np.arange(case.q.shape[0] * case.num_heads, dtype=np.int64)
    ref_o, ref_l = oracle_rows(case, rows, "long_185k/all")
    o, l, st = run_full(case, kernel)
    assert st == 0
    compare(o.reshape(-1, o.shape[-1]), l.reshape(-1), ref_o, ref_l, f"{kernel}/long_185k every row")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["tree_32k", "sweep_q4"])
def test_full_unit_every_row(name):
    """Every row of one full 256-row unit (row block 0) of every sequence, tensor-core path."""
    case = full_case(name)
    rows = unit_rows(case)
    ref_o, ref_l = oracle_rows(case, rows, f"{name}/unit0")
    o, l, st = run_full(case, "tc")
    assert st == 0
    compare(o.reshape(-1, o.shape[-1])[rows], l.reshape(-1)[rows], ref_o, ref_l, f"tc/{name} unit rows")
