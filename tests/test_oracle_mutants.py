"""Plausible mistakes planted in the oracle (on the CPU) must break a pin.

Each mutant is a one-place edit of the oracle's C source (a dropped term, a
wrong index or bound, a missing normalisation), compiled into a temporary
library.  The battery below reuses the pins of test_oracle_pins.py; a mutant
that passes all of them would mean the pins cannot tell that mistake from the
definition.  Nothing here touches a GPU.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth
from tests import test_oracle_pins as pins

MUTANTS = {
    "drop_scale": ("s *= P->sm_scale;", "s *= 1.0;"),
    "no_max_subtraction": ("double w = exp(s - m);", "double w = exp(s);"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "value_dims_shifted": ("out[d] += w * bf16_to_f64(row[d]);", "out[d] += w * bf16_to_f64(row[d + 64]);"),
    "score_over_latent_only": ("for (int d = 0; d < ORACLE_DQK; ++d) s += qd[d] * bf16_to_f64(row[d]);",
                               "for (int d = 0; d < ORACLE_DV; ++d) s += qd[d] * bf16_to_f64(row[d]);"),
    "causal_excludes_self": ("for (int k = 0; k <= i; ++k) m |= 1ULL << k;", "for (int k = 0; k < i; ++k) m |= 1ULL << k;"),
    "prefix_off_by_one": ("int visible = (j < prefix) ||", "int visible = (j <= prefix) ||"),
    "parent_ignored": ("      k = p;\n", "      k = -1;\n"),
    "no_normalisation": ("out[d] /= l;", "out[d] /= 1.0;"),
    "index_without_sequence_offset": ("int64_t slot = P->kv_indices[kv0 + j];", "int64_t slot = P->kv_indices[j];"),
    "head_ignored": ("((int64_t)t * P->num_heads + h) * ORACLE_DQK", "((int64_t)t * P->num_heads) * ORACLE_DQK"),
    "merge_lse_without_max": ("      *lse = mx + log(z);\n", "      *lse = log(z);\n"),
    "merge_weight_unnormalised": ("double w = exp(l_s[s] - *lse);", "double w = exp(l_s[s] - mx);"),
    "split_bounds_overlap": ("hi = (int)(((int64_t)n_kv * (s + 1)) / S);", "hi = (int)(((int64_t)n_kv * (s + 1)) / S) + 1;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(oracle.SRC).read()
    assert src.count(old) == 1, f"mutant {name}: pattern must occur exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    return oracle.lib(str(so))


def _battery(L):
    """Yield (pin name, passed) for a fast subset of the pins, run on library L."""
    cases = [pins.small_case(13, [7, 2], [4, 1]),
             pins.small_case(14, [6, 3], [4, 4], tree=2),
             pins.small_case(17, [9, 0], [3, 5], heads=3)]
    for k, case in enumerate(cases):
        try:
            out, lse = oracle.verify(case, lib_=L)
            ro, rl = pins.library_attention(case)
            yield f"sdpa{k}", bool(np.allclose(out, ro, atol=1e-9, rtol=0) and np.allclose(lse, rl, atol=1e-9, rtol=0))
        except ValueError:
            yield f"sdpa{k}", False
    # explicit visibility in which some queries do not see draft 0
    case = pins.small_case(16, [4, 6], [4, 3])
    dm = np.array([0b0001, 0b0010, 0b0110, 0b1101, 0b001, 0b110, 0b100], dtype=np.uint64)
    try:
        out, lse = oracle.verify(case, draft_mask=dm, lib_=L)
        ro, rl = pins.library_attention(case, draft_mask=dm)
        yield "sdpa_mask", bool(np.allclose(out, ro, atol=1e-9, rtol=0) and np.allclose(lse, rl, atol=1e-9, rtol=0))
    except ValueError:
        yield "sdpa_mask", False
    case, rows = pins.designed_case(1000.0, [0.0, -1.0, -3.0])
    out, lse = oracle.verify(case, lib_=L)
    w = np.array([1.0, math.exp(-1.0), math.exp(-3.0)])
    expect = (w[:, None] * rows[:, :512]).sum(0) / w.sum()
    ok = np.all(np.isfinite(out)) and np.allclose(out[0, 0], expect, atol=1e-9) and \
        abs(lse[0, 0] - (1000.0 + math.log(w.sum()))) < 1e-9
    yield "large_scores", bool(ok)
    case = pins.small_case(41, [30, 3, 12], [4, 2, 5], heads=2, tree=3)
    o1, l1 = oracle.verify(case, lib_=L)
    for s in (2, 7):
        o2, l2 = oracle.verify_split(case, s, lib_=L)
        yield f"split{s}", bool(np.allclose(o1, o2, atol=1e-12, rtol=0) and np.allclose(l1, l2, atol=1e-12, rtol=0))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    L = _build_mutant(tmp_path, name, old, new)
    results = dict(_battery(L))
    assert not all(results.values()), f"mutant {name} passed every pin: {results}"


def test_unmutated_passes_battery():
    results = dict(_battery(oracle.lib()))
    assert all(results.values()), results


# ---------------------------------------------------------------- tree acceptance (Python oracle)

ACCEPT_MUTANTS = {
    "expects_own_target": ("expected = root_token[b] if p < 0 else target_token[q0 + p]",
                           "expected = root_token[b] if p < 0 else target_token[q0 + i]"),
    "parent_acceptance_ignored": ("accepted[i] = (p < 0 or accepted[p]) and", "accepted[i] = True and"),
    "ties_to_larger_index": ("depth[i] > depth[best]", "depth[i] >= depth[best]"),
    "next_after_parent": ("next_token[b] = target_token[q0 + best]",
                          "next_token[b] = target_token[q0 + max(par[best], 0)]"),
    "depth_not_accumulated": ("depth[i] = 0 if p < 0 else depth[p] + 1", "depth[i] = 0 if p < 0 else 1"),
}


def _accept_mutant(old, new):
    import inspect
    from typing import Optional
    src = inspect.getsource(oracle.tree_accept)
    assert src.count(old) == 1, f"pattern must occur exactly once: {old}"
    ns = {"np": np, "Optional": Optional}
    exec(src.replace(old, new), ns)
    return ns["tree_accept"]


@pytest.mark.parametrize("name", sorted(ACCEPT_MUTANTS))
def test_tree_accept_mutant_breaks_a_pin(name, monkeypatch):
    mutant = _accept_mutant(*ACCEPT_MUTANTS[name])
    monkeypatch.setattr(oracle, "tree_accept", mutant)
    failed = []
    for pin in (pins.test_tree_accept_hand_worked, pins.test_tree_accept_empty_sequences_and_parent_none_is_chain,
                pins.test_tree_accept_matches_brute_force_on_random_trees):
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every tree-acceptance pin"
