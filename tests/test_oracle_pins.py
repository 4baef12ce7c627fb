"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties the oracle to an independent source of truth:
  * a library routine (torch's scaled_dot_product_attention in float64, scipy's
    logsumexp, networkx ancestor sets) on small dense cases;
  * closed forms (a single visible key, equal scores, designed score sets, a
    two-part merge);
  * invariants of the definition (slot permutation, split-and-merge, shifting
    every score by a constant, a parent chain equal to the causal mask).
test_oracle_mutants.py checks that plausible mistakes in the oracle break at
least one of these.
"""
import math

import networkx as nx
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from speculative_decoding_mla_gb300 import synth

D_QK, D_V = 576, 512


def bf16(x):
    return synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def widen(b):
    return synth.bf16_bits_to_f64(b)


# ---------------------------------------------------------------- library pin

def visibility_library(case, draft_mask=None):
    """Per sequence: bool [Q_b, Q_b] visibility of draft keys, derived without the oracle:
    explicit bits, networkx ancestors for a tree, numpy tril for causal."""
    out = []
    for b in range(case.batch):
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        n = q1 - q0
        if draft_mask is not None:
            m = np.array([[(int(draft_mask[q0 + i]) >> k) & 1 for k in range(n)] for i in range(n)], dtype=bool)
        elif case.parent is not None:
            g = nx.DiGraph()
            g.add_nodes_from(range(n))
            for i in range(n):
                p = int(case.parent[q0 + i])
                if p >= 0:
                    g.add_edge(p, i)
            m = np.zeros((n, n), dtype=bool)
            for i in range(n):
                for a in nx.ancestors(g, i) | {i}:
                    m[i, a] = True
        else:
            m = np.tril(np.ones((n, n), dtype=bool))
        out.append(m)
    return out


def library_attention(case, draft_mask=None):
    """Dense masked attention through torch SDPA (float64, CPU) and scipy logsumexp."""
    H = case.num_heads
    T = case.q.shape[0]
    out = np.zeros((T, H, D_V))
    lse = np.zeros((T, H))
    vis = visibility_library(case, draft_mask)
    qf = widen(case.q)
    pool = widen(case.kv_pool)
    for b in range(case.batch):
        k0, k1 = int(case.kv_indptr[b]), int(case.kv_indptr[b + 1])
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        n_q, n_kv = q1 - q0, k1 - k0
        P = n_kv - n_q
        rows = pool[case.kv_indices[k0:k1]]                   # [N, 576]
        mask = np.zeros((n_q, n_kv), dtype=bool)
        mask[:, :P] = True
        mask[:, P:] = vis[b]
        for h in range(H):
            Q = torch.from_numpy(qf[q0:q1, h, :].copy())
            K = torch.from_numpy(rows.copy())
            V = torch.from_numpy(rows[:, :D_V].copy())
            o = torch.nn.functional.scaled_dot_product_attention(
                Q[None], K[None], V[None], attn_mask=torch.from_numpy(mask)[None], scale=case.sm_scale)[0]
            out[q0:q1, h] = o.numpy()
            sc = case.sm_scale * (qf[q0:q1, h, :] @ rows.T)
            lse[q0:q1, h] = scipy.special.logsumexp(sc, b=mask.astype(np.float64), axis=-1)
    return out, lse


def small_case(seed, prefixes, drafts, heads=2, tree=None, permute=True, pool_extra=5):
    pool = sum(prefixes) + (sum(drafts) if not isinstance(drafts, int) else drafts * len(prefixes)) + pool_extra
    return synth.make_case("small", prefixes, drafts, num_heads=heads, pool_slots=pool, permute=permute,
                           tree_depth=tree, seed=seed)


@pytest.mark.parametrize("seed,prefixes,drafts,tree", [
    (11, [8], 4, None),
    (12, [0, 5], [3, 2], None),
    (13, [7, 2], [4, 1], None),
    (14, [6, 3], [4, 4], 2),
    (15, [1], 1, None),
])
def test_library_sdpa(seed, prefixes, drafts, tree):
    case = small_case(seed, prefixes, drafts, tree=tree)
    out, lse = oracle.verify(case)
    ref_o, ref_l = library_attention(case)
    np.testing.assert_allclose(out, ref_o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, ref_l, atol=1e-12, rtol=0)


def test_library_sdpa_explicit_mask():
    case = small_case(16, [4, 6], [4, 3])
    rng = np.random.default_rng(0)
    dm = []
    for b in range(case.batch):
        n = int(case.qo_indptr[b + 1] - case.qo_indptr[b])
        for i in range(n):
            bits = int(rng.integers(0, 1 << n)) | (1 << i)
            dm.append(bits)
    dm = np.array(dm, dtype=np.uint64)
    out, lse = oracle.verify(case, draft_mask=dm)
    ref_o, ref_l = library_attention(case, draft_mask=dm)
    np.testing.assert_allclose(out, ref_o, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, ref_l, atol=1e-12, rtol=0)


# ---------------------------------------------------------------- closed forms

def hand_case(q_rows, kv_rows, prefix, sm_scale, draft_mask=None, parent=None):
    """One sequence, one head: q_rows [Q,576], kv_rows [N,576] (float values exact in bf16)."""
    q = bf16(np.asarray(q_rows, dtype=np.float64)).reshape(len(q_rows), 1, D_QK)
    kv = bf16(np.asarray(kv_rows, dtype=np.float64)).reshape(len(kv_rows), D_QK)
    assert np.array_equal(widen(q).reshape(len(q_rows), D_QK), np.asarray(q_rows, dtype=np.float64))
    assert np.array_equal(widen(kv), np.asarray(kv_rows, dtype=np.float64))
    n = len(kv_rows)
    nq = len(q_rows)
    assert prefix == n - nq
    return synth.Case(name="hand", q=q, kv_pool=kv, kv_indptr=np.array([0, n], np.int32),
                      kv_indices=np.arange(n, dtype=np.int32), qo_indptr=np.array([0, nq], np.int32),
                      parent=None if parent is None else np.asarray(parent, np.int32), sm_scale=sm_scale)


def int_row(rng, lo=-4, hi=5):
    return rng.integers(lo, hi, size=D_QK).astype(np.float64)


def test_single_visible_key_exact():
    rng = np.random.default_rng(1)
    q = int_row(rng)
    k = int_row(rng)
    case = hand_case([q], [k], 0, 0.125)
    out, lse = oracle.verify(case)
    # one visible key: softmax weight exactly 1, so out is that key's latent row
    assert np.array_equal(out[0, 0], k[:D_V])
    s_exact = 0.125 * float(int(np.dot(q.astype(np.int64), k.astype(np.int64))))
    assert lse[0, 0] == s_exact


def test_equal_scores_give_mean_and_log_count():
    rng = np.random.default_rng(2)
    rows = [rng.normal(size=D_QK) for _ in range(9)]
    rows = [widen(bf16(r)) for r in rows]
    qs = [np.zeros(D_QK) for _ in range(3)]
    case = hand_case(qs, rows, 6, 0.3)
    out, lse = oracle.verify(case)
    R = np.array(rows)
    for i in range(3):
        visible = R[: 6 + i + 1]
        np.testing.assert_allclose(out[i, 0], visible[:, :D_V].mean(axis=0), atol=1e-13, rtol=0)
        assert abs(lse[i, 0] - math.log(len(visible))) < 1e-15


def test_zero_scale_gives_mean():
    case = small_case(21, [5, 3], [2, 3])
    case.sm_scale = 0.0
    out, lse = oracle.verify(case)
    pool = widen(case.kv_pool)
    for b in range(case.batch):
        k0, k1 = int(case.kv_indptr[b]), int(case.kv_indptr[b + 1])
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        P = (k1 - k0) - (q1 - q0)
        rows = pool[case.kv_indices[k0:k1]]
        for i in range(q1 - q0):
            vis = rows[: P + i + 1, :D_V]
            for h in range(case.num_heads):
                np.testing.assert_allclose(out[q0 + i, h], vis.mean(axis=0), atol=1e-13, rtol=0)
                assert abs(lse[q0 + i, h] - math.log(P + i + 1)) < 1e-14


def designed_case(base, deltas):
    """Keys whose scores are exactly base + deltas[j]: q = e_0 + e_1, key j has
    element 0 = base and element 1 = deltas[j] (all exact in bf16), sm_scale = 1.
    The last key is the single causal draft, the rest prefix."""
    rng = np.random.default_rng(3)
    q = np.zeros(D_QK)
    q[0] = q[1] = 1.0
    rows = []
    for d in deltas:
        r = widen(bf16(rng.normal(size=D_QK)))
        r[0] = base
        r[1] = d
        rows.append(r)
    return hand_case([q], rows, len(deltas) - 1, 1.0), np.array(rows)


def test_closed_form_three_keys():
    case, rows = designed_case(0.0, [0.0, 1.0, 2.0])
    out, lse = oracle.verify(case)
    w = np.array([1.0, math.e, math.e ** 2])
    expect = (w[:, None] * rows[:, :D_V]).sum(0) / w.sum()
    np.testing.assert_allclose(out[0, 0], expect, atol=1e-13, rtol=0)
    assert abs(lse[0, 0] - math.log(1 + math.e + math.e ** 2)) < 1e-14


@pytest.mark.parametrize("base", [1000.0, -1000.0, 80.0])
def test_large_scores_closed_form(base):
    # scores far beyond exp's range: only a max-subtracted evaluation survives
    case, rows = designed_case(base, [0.0, -1.0, -3.0])
    out, lse = oracle.verify(case)
    w = np.array([1.0, math.exp(-1.0), math.exp(-3.0)])
    expect = (w[:, None] * rows[:, :D_V]).sum(0) / w.sum()
    np.testing.assert_allclose(out[0, 0], expect, atol=1e-12, rtol=0)
    assert abs(lse[0, 0] - (base + math.log(w.sum()))) < 1e-12 * max(1.0, abs(base))


def test_no_visible_key():
    rng = np.random.default_rng(4)
    case = hand_case([int_row(rng)], [int_row(rng)], 0, 0.1)
    out, lse = oracle.verify(case, draft_mask=np.array([0], np.uint64))
    assert np.all(out == 0.0) and lse[0, 0] == -math.inf


# ---------------------------------------------------------------- invariants

def test_permutation_invariance_bitwise():
    case = small_case(31, [9, 4, 0], [3, 4, 2], heads=3)
    out, lse = oracle.verify(case)
    S = case.pool_slots
    pi = synth.permutation(99, synth.TAG_AUX, S)
    pool2 = np.empty_like(case.kv_pool)
    pool2[pi] = case.kv_pool
    case2 = synth.Case(name="perm", q=case.q, kv_pool=pool2, kv_indptr=case.kv_indptr,
                       kv_indices=pi[case.kv_indices].astype(np.int32), qo_indptr=case.qo_indptr,
                       sm_scale=case.sm_scale)
    out2, lse2 = oracle.verify(case2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("splits", [1, 2, 7, 40])
def test_split_merge_identity(splits):
    case = small_case(41, [30, 3, 12], [4, 2, 5], heads=2, tree=3)
    out, lse = oracle.verify(case)
    o2, l2 = oracle.verify_split(case, splits)
    np.testing.assert_allclose(o2, out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l2, lse, atol=1e-12, rtol=0)


def test_parent_chain_equals_causal():
    case = small_case(51, [6, 2], [5, 3], heads=2)
    out, lse = oracle.verify(case)
    chain = np.concatenate([np.arange(-1, 4), np.arange(-1, 2)]).astype(np.int32)
    case.parent = chain
    o2, l2 = oracle.verify(case)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_score_shift_through_rope_column():
    # pool column 575 (rope) set to 1 in every row; q[:, :, 575] = 0 vs 2:
    # every score moves by 2 * sm_scale, the output stays, the lse moves by the same
    case = small_case(61, [7, 3], [3, 2], heads=2)
    one = bf16(np.array([1.0]))[0]
    two = bf16(np.array([2.0]))[0]
    case.kv_pool[:, 575] = one
    case.q[:, :, 575] = 0
    out, lse = oracle.verify(case)
    case.q[:, :, 575] = two
    o2, l2 = oracle.verify(case)
    np.testing.assert_allclose(o2, out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(l2 - lse, 2.0 * case.sm_scale, atol=1e-12, rtol=0)


# ---------------------------------------------------------------- merge and masks on their own

def test_merge_closed_form():
    o_parts = np.zeros((3, 2, 4))
    o_parts[0, 0] = [1, 0, 0, 0]
    o_parts[1, 0] = [0, 1, 0, 0]
    o_parts[2, 0] = [5, 5, 5, 5]
    lse_parts = np.array([[0.0, -math.inf], [math.log(3.0), -math.inf], [-math.inf, -math.inf]])
    o, lse = oracle.merge(o_parts, lse_parts)
    np.testing.assert_allclose(o[0], [0.25, 0.75, 0, 0], atol=1e-15)
    assert abs(lse[0] - math.log(4.0)) < 1e-15
    assert np.all(o[1] == 0) and lse[1] == -math.inf


def test_tree_masks_match_graph_ancestors():
    parents = [synth.tree_parents(7, 64, 8, s) for s in range(5)]
    qo = np.zeros(6, np.int32)
    qo[1:] = np.cumsum([64] * 5)
    masks = oracle.tree_masks(np.concatenate(parents), qo)
    for s, par in enumerate(parents):
        g = nx.DiGraph()
        g.add_nodes_from(range(64))
        for i, p in enumerate(par):
            if p >= 0:
                g.add_edge(int(p), i)
        depth = nx.shortest_path_length(g, 0)
        assert max(depth.values()) <= 8
        for i in range(64):
            bits = sum(1 << a for a in nx.ancestors(g, i) | {i})
            assert int(masks[s * 64 + i]) == bits


def test_sampled_rows_equal_full():
    case = small_case(71, [20, 11], [4, 6], heads=3)
    out, lse = oracle.verify(case)
    rows = np.array([0, 5, 7, 12, 29], dtype=np.int64)
    o, l = oracle.verify_rows(case, rows)
    H = case.num_heads
    for k, r in enumerate(rows):
        assert np.array_equal(o[k], out[r // H, r % H]) and l[k] == lse[r // H, r % H]


def test_thread_count_does_not_change_any_row():
    """Rows are independent: every split of the rows over threads gives the same bits (a row skipped
    or computed twice at a thread boundary would show here)."""
    case = small_case(73, [37, 0, 12, 5], [7, 3, 1, 8], heads=5)
    out1, lse1 = oracle.verify(case, threads=1)
    for threads in (2, 3, 7, 64):
        out, lse = oracle.verify(case, threads=threads)
        assert np.array_equal(out, out1) and np.array_equal(lse, lse1)


def test_rejects_bad_inputs():
    case = small_case(81, [3], 2, heads=1)
    bad = synth.Case(name="bad", q=case.q, kv_pool=case.kv_pool, kv_indptr=case.kv_indptr,
                     kv_indices=np.full_like(case.kv_indices, case.pool_slots), qo_indptr=case.qo_indptr)
    with pytest.raises(ValueError):
        oracle.verify(bad)
    with pytest.raises(ValueError):
        oracle.tree_masks(np.array([-1, 1], np.int32), np.array([0, 2], np.int32))


# ---------------------------------------------------------------- tree acceptance

def _accept_one(parent, draft, target, root):
    qo = np.array([0, len(draft)])
    par = None if parent is None else np.array(parent, np.int32)
    return oracle.tree_accept(qo, par, np.array(draft, np.int32), np.array(target, np.int32),
                              np.array([root], np.int32))


def test_tree_accept_hand_worked():
    # chain, every draft matches the target's token after its predecessor
    n, path, nxt, bad = _accept_one(None, [10, 11, 12, 13], [11, 12, 13, 14], 10)
    assert n[0] == 4 and list(path) == [0, 1, 2, 3] and nxt[0] == 14 and not bad[0]
    # chain, the first draft is already wrong: nothing accepted, the prefix's token is next
    n, path, nxt, _ = _accept_one(None, [9, 11, 12, 13], [11, 12, 13, 14], 10)
    assert n[0] == 0 and list(path) == [-1] * 4 and nxt[0] == 10
    # chain, wrong at the third node: two accepted, the second node's target token is next
    n, path, nxt, _ = _accept_one(None, [10, 11, 99, 13], [11, 12, 13, 14], 10)
    assert n[0] == 2 and list(path) == [0, 1, -1, -1] and nxt[0] == 12
    # tree: roots 0 and 1 (only 1 matches the prefix's token 5), 2 under 1 matches, 3 under 0 would
    # match its parent's token but 0 was rejected, 4 under 2 is wrong
    parent = [-1, -1, 1, 0, 2]
    draft = [4, 5, 7, 8, 0]
    target = [8, 7, 6, 1, 2]
    n, path, nxt, _ = _accept_one(parent, draft, target, 5)
    assert n[0] == 2 and list(path) == [1, 2, -1, -1, -1] and nxt[0] == 6
    # equal depths: the smaller index wins (nodes 1 and 2 are both accepted children of 0)
    n, path, nxt, _ = _accept_one([-1, 0, 0], [3, 4, 4], [4, 9, 8], 3)
    assert n[0] == 2 and list(path) == [0, 1, -1] and nxt[0] == 9
    # a deeper accepted node beats a shallower one with a smaller index
    n, path, nxt, _ = _accept_one([-1, 0, 0, 2], [3, 4, 4, 8], [4, 9, 8, 1], 3)
    assert n[0] == 3 and list(path) == [0, 2, 3, -1] and nxt[0] == 1
    # malformed parent (a parent after its child): flagged, nothing accepted
    n, path, nxt, bad = _accept_one([-1, 2, 0], [3, 4, 4], [4, 9, 8], 3)
    assert bad[0] and n[0] == 0 and nxt[0] == 3


def test_tree_accept_empty_sequences_and_parent_none_is_chain():
    qo = np.array([0, 0, 3, 3])
    draft = np.array([7, 8, 1], np.int32)
    target = np.array([8, 2, 5], np.int32)
    root = np.array([1, 7, 4], np.int32)
    n, path, nxt, bad = oracle.tree_accept(qo, None, draft, target, root)
    assert list(n) == [0, 2, 0] and list(nxt) == [1, 2, 4] and not bad.any()
    n2, path2, nxt2, _ = oracle.tree_accept(qo, np.array([-1, 0, 1], np.int32), draft, target, root)
    assert np.array_equal(n, n2) and np.array_equal(path, path2) and np.array_equal(nxt, nxt2)


def _brute_force_accept(parent, draft, target, root):
    """Every root-to-node path, accepted when each token equals the target's token after its
    predecessor; the longest accepted path, ties by the smaller last node."""
    n = len(draft)
    best = []
    for end in range(n):
        path = [end]
        while parent[path[-1]] >= 0:
            path.append(parent[path[-1]])
        path.reverse()
        prev_tok = root
        ok = True
        for node in path:
            if draft[node] != prev_tok:
                ok = False
                break
            prev_tok = target[node]
        if ok and len(path) > len(best):
            best = path
    return best, (target[best[-1]] if best else root)


def test_tree_accept_matches_brute_force_on_random_trees():
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(1, 20))
        parent = synth.tree_parents(trial, n, int(rng.integers(1, 8)), 0)
        target = rng.integers(0, 4, n).astype(np.int32)
        root = int(rng.integers(0, 4))
        # drafts that often (not always) follow the target, so paths of every length occur
        draft = np.empty(n, np.int32)
        for i in range(n):
            follow = root if parent[i] < 0 else target[parent[i]]
            draft[i] = follow if rng.random() < 0.7 else int(rng.integers(0, 4))
        path, nxt = _brute_force_accept(list(parent), list(draft), list(target), root)
        n_acc, p_acc, nxt_acc, bad = _accept_one(parent, draft, target, root)
        assert not bad[0]
        assert n_acc[0] == len(path) and list(p_acc[:len(path)]) == path and nxt_acc[0] == nxt
        assert (p_acc[len(path):] == -1).all()


# ---------------------------------------------------------------- fp8 (e4m3) storage

def test_e4m3_values_match_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert oracle.e4m3_value(np.array([0x7E], np.uint8))[0] == 448.0
    assert oracle.e4m3_value(np.array([0x01], np.uint8))[0] == 2.0 ** -9


def test_dequantize_e4m3_rounds_to_nearest_even():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, 4096).astype(np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    for scale in (1.0, 0.0037, 1.0 / 3.0, 2.0 ** -5):
        bits = oracle.dequantize_e4m3(codes, scale)
        # the product in float32, then float32 -> bf16 by torch (round to nearest even)
        prod = torch.from_numpy(oracle.e4m3_value(codes).astype(np.float32)) * torch.tensor(scale, dtype=torch.float32)
        ref = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(bits, ref)
    # a tie: 1 + 2^-8 is halfway between two bf16 values and goes to the even one (1.0)
    tie = np.array([1.0 + 2.0 ** -8], np.float32)
    assert oracle._bf16_rne_bits(tie)[0] == 0x3F80
