"""GPU parity of the tree-acceptance kernel with the oracle (integer results:
exact equality), on random trees and chains, empty sequences and malformed
parents."""
import numpy as np
import pytest

import oracle
from speculative_decoding_mla_gb300 import synth

pytestmark = pytest.mark.gpu


def _mods():
    import torch
    from speculative_decoding_mla_gb300 import build as vbuild
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding
    return torch, binding


def _batch(seed, B, chain=False, follow=0.75, vocab=5):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 65, B)
    counts[rng.integers(0, B)] = 64
    counts[rng.integers(0, B)] = 0
    qo = np.zeros(B + 1, np.int32)
    qo[1:] = np.cumsum(counts)
    T = int(qo[-1])
    parent = np.empty(T, np.int32)
    for b in range(B):
        n = int(counts[b])
        if n:
            parent[qo[b]:qo[b + 1]] = (np.arange(n) - 1 if chain
                                       else synth.tree_parents(seed + b, n, int(rng.integers(1, 9)), b))
    target = rng.integers(0, vocab, T).astype(np.int32)
    root = rng.integers(0, vocab, B).astype(np.int32)
    draft = np.empty(T, np.int32)
    for b in range(B):
        for i in range(int(counts[b])):
            p = parent[qo[b] + i]
            want = root[b] if p < 0 else target[qo[b] + p]
            draft[qo[b] + i] = want if rng.random() < follow else int(rng.integers(0, vocab))
    return qo, parent, draft, target, root


def _run(qo, parent, draft, target, root):
    torch, binding = _mods()
    B, T = len(qo) - 1, int(qo[-1])
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((max(T, 1),), -7, dtype=torch.int32, device="cuda")[:T]
    nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    binding.verify_attn_mla_tree_accept(d(qo), d(parent) if parent is not None else None, d(draft), d(target), d(root),
                                        acc, path, nxt, st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), nxt.cpu().numpy(), int(st[0]), int(st[1])


@pytest.mark.parametrize("chain", [False, True])
def test_tree_accept_matches_oracle(chain):
    for seed in (1, 2, 3):
        qo, parent, draft, target, root = _batch(100 * seed + int(chain), 37, chain=chain)
        ref = oracle.tree_accept(qo, parent, draft, target, root)
        acc, path, nxt, st, _ = _run(qo, parent, draft, target, root)
        assert st == 0
        assert np.array_equal(acc, ref[0]) and np.array_equal(path, ref[1]) and np.array_equal(nxt, ref[2])
        assert ref[0].max() >= 3  # some long paths occur


def test_tree_accept_without_parents_is_the_chain():
    qo, parent, draft, target, root = _batch(7, 20, chain=True)
    a1 = _run(qo, parent, draft, target, root)
    a2 = _run(qo, None, draft, target, root)
    assert all(np.array_equal(x, y) for x, y in zip(a1[:3], a2[:3]))


def test_tree_accept_malformed_parent_is_reported():
    _, binding = _mods()
    qo, parent, draft, target, root = _batch(9, 6)
    b = int(np.argmax(np.diff(qo) >= 3))
    parent = parent.copy()
    parent[qo[b] + 2] = 2  # a node that is its own parent
    ref = oracle.tree_accept(qo, parent, draft, target, root)
    acc, path, nxt, st, info = _run(qo, parent, draft, target, root)
    assert ref[3][b] and st == binding.VMLA_ERR_PARENT and info == b
    assert np.array_equal(acc, ref[0]) and np.array_equal(nxt, ref[2]) and np.array_equal(path, ref[1])
