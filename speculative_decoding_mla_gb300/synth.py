"""Seeded synthetic inputs for MLA speculative-decoding verify attention.

This module draws the random inputs only: it holds none of the attention
arithmetic, no mask logic and no planning, so that both the CPU oracle and the
GPU path can take their inputs from it without sharing any of the method.

Generator (every value is reproducible from (seed, stream tag, index)):
  * splitmix64 as a counter-based generator: the i-th 64-bit word of a stream
    is mix(base + (i + 1) * 0x9E3779B97F4A7C15), with mix the splitmix64
    finaliser (xor-shift 30 / multiply / xor-shift 27 / multiply / xor-shift 31)
    and base = mix(seed * 0x9E3779B97F4A7C15 + tag);
  * uniforms u = ((word >> 11) + 0.5) * 2**-53, strictly inside (0, 1);
  * normals by Box-Muller, two per pair of uniforms: r = sqrt(-2 ln u1),
    z0 = r cos(2 pi u2), z1 = r sin(2 pi u2);
  * values rounded once f64 -> f32 (round-to-nearest-even) and then f32 ->
    bf16 (round-to-nearest-even on the bit pattern), stored as uint16 bits.

Workload shapes follow the verify step described in "The Build That Bridged
Design and Deployment", section "What This Build Achieves: The paged+bf16
Kernel": a segmented batch of requests, each a prefix read through a slot
indirection (page_size = 1) plus a small block or tree of draft positions.
The dimensions (64 heads, 576 = 512 latent + 64 rope per token, sm_scale =
1/sqrt(192)) and the five named workloads are those of the target shapes.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

D_QK = 576
D_V = 512
NUM_HEADS = 64
SM_SCALE = 1.0 / math.sqrt(192.0)

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream tags, one per kind of draw
TAG_Q = 1
TAG_KV = 2
TAG_PERM = 3
TAG_LEN = 4
TAG_TREE = 5
TAG_AUX = 6

_U64 = 0xFFFFFFFFFFFFFFFF


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _load_gen():
    """Compile (when stale) and load the C generator beside this file."""
    global _GEN
    if _GEN is not None:
        return _GEN
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "synth_gen.c")
    lib = os.path.join(here, "_synth_gen.so")
    if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        tmp = f"{lib}.{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"])
        os.replace(tmp, lib)
    g = ctypes.CDLL(lib)
    u64, i64 = ctypes.c_uint64, ctypes.c_int64
    g.synth_words.argtypes = [u64, u64, u64, i64, ctypes.c_void_p]
    g.synth_normals_f64.argtypes = [u64, u64, i64, i64, ctypes.c_double, ctypes.c_void_p]
    g.synth_bf16_normals.argtypes = [u64, u64, i64, i64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
    for f in (g.synth_words, g.synth_normals_f64, g.synth_bf16_normals):
        f.restype = None
    _GEN = g
    return g


_GEN = None


def words(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """The n 64-bit words [offset, offset + n) of stream (seed, tag)."""
    out = np.empty(n, dtype=np.uint64)
    if n:
        _load_gen().synth_words(seed & _U64, tag, offset, n, out.ctypes.data)
    return out


def words_numpy(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """Same words as words(), computed with numpy (slow; used to check the C generator)."""
    with np.errstate(over="ignore"):
        s = np.array([np.uint64(seed & _U64) * _GOLDEN + np.uint64(tag)], dtype=np.uint64)
        base = _mix(s)[0]
        idx = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix(base + idx * _GOLDEN)


def uniforms(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    w = words(seed, tag, n, offset)
    return ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normals(seed: int, tag: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """n standard normals (times sigma) in float64, Box-Muller on stream (seed, tag)."""
    out = np.empty(n, dtype=np.float64)
    if n:
        _load_gen().synth_normals_f64(seed & _U64, tag, 0, n, sigma, out.ctypes.data)
    return out


def normals_numpy(seed: int, tag: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """Same normals as normals(), computed with numpy (used to check the C generator)."""
    p1 = (n + 1) // 2
    w = words_numpy(seed, tag, 2 * p1)
    u = ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = 2.0 * np.pi * u[1::2]
    z = np.empty(2 * p1, dtype=np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return z[:n] * sigma


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_normals(seed: int, tag: int, n: int, sigma: float) -> np.ndarray:
    """n normals times sigma, rounded to bf16, as uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load_gen().synth_bf16_normals(seed & _U64, tag, 0, n, sigma, out.ctypes.data, os.cpu_count() or 1)
    return out


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (argsort of n iid 64-bit words, ties by position)."""
    w = words(seed, tag, n)
    return np.argsort(w, kind="stable").astype(np.int32)


def tree_parents(seed: int, n_nodes: int, max_depth: int, seq: int) -> np.ndarray:
    """Draft-tree parents for one sequence: node 0 is the root (parent -1, depth 0);
    node i >= 1 takes its parent uniformly from the earlier nodes whose depth is
    below max_depth, so no node is deeper than max_depth."""
    parent = np.full(n_nodes, -1, dtype=np.int32)
    depth = np.zeros(n_nodes, dtype=np.int32)
    w = words(seed, TAG_TREE, n_nodes, offset=seq * 4096)
    for i in range(1, n_nodes):
        eligible = [p for p in range(i) if depth[p] < max_depth]
        k = int(w[i] % np.uint64(len(eligible)))
        parent[i] = eligible[k]
        depth[i] = depth[parent[i]] + 1
    return parent


@dataclass
class Case:
    """One verify-attention call's inputs (host arrays; bf16 as uint16 bits).

    Sequence b owns kv_indices[kv_indptr[b]:kv_indptr[b+1]] (N_b slots, the last
    Q_b of them holding the draft tokens' rows) and query rows
    qo_indptr[b]..qo_indptr[b+1] (Q_b draft positions).  parent, when present,
    holds each draft node's local parent index (-1 for a root); when absent the
    drafts are causal among themselves."""
    name: str
    q: np.ndarray            # [T_q, H, 576] uint16
    kv_pool: np.ndarray      # [S, 576] uint16
    kv_indptr: np.ndarray    # [B+1] int32
    kv_indices: np.ndarray   # [sum N_b] int32
    qo_indptr: np.ndarray    # [B+1] int32
    parent: Optional[np.ndarray] = None   # [T_q] int32 or None
    sm_scale: float = SM_SCALE
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.kv_indptr) - 1

    @property
    def num_heads(self) -> int:
        return self.q.shape[1]

    @property
    def pool_slots(self) -> int:
        return self.kv_pool.shape[0]

    @property
    def prefix_lens(self) -> np.ndarray:
        return np.diff(self.kv_indptr) - np.diff(self.qo_indptr)


def make_case(name: str, prefixes, drafts, *, num_heads: int = NUM_HEADS, pool_slots: Optional[int] = None,
              permute: bool = True, tree_depth: Optional[int] = None, seed: int = 0,
              q_sigma: float = 1.0, kv_sigma: float = 0.5, sm_scale: float = SM_SCALE) -> Case:
    prefixes = [int(p) for p in prefixes]
    if isinstance(drafts, int):
        drafts = [drafts] * len(prefixes)
    drafts = [int(d) for d in drafts]
    B = len(prefixes)
    n_kv = [p + d for p, d in zip(prefixes, drafts)]
    kv_indptr = np.zeros(B + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(n_kv)
    qo_indptr = np.zeros(B + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(drafts)
    total_kv = int(kv_indptr[-1])
    S = total_kv if pool_slots is None else int(pool_slots)
    assert S >= total_kv
    if permute:
        kv_indices = permutation(seed, TAG_PERM, S)[:total_kv].copy()
    else:
        kv_indices = np.arange(total_kv, dtype=np.int32)
    T_q = int(qo_indptr[-1])
    q = bf16_normals(seed, TAG_Q, T_q * num_heads * D_QK, q_sigma).reshape(T_q, num_heads, D_QK)
    kv_pool = bf16_normals(seed, TAG_KV, S * D_QK, kv_sigma).reshape(S, D_QK)
    parent = None
    if tree_depth is not None:
        parent = np.concatenate([tree_parents(seed, d, tree_depth, b) for b, d in enumerate(drafts)]).astype(np.int32)
    return Case(name=name, q=q, kv_pool=kv_pool, kv_indptr=kv_indptr, kv_indices=kv_indices,
                qo_indptr=qo_indptr, parent=parent, sm_scale=sm_scale,
                meta=dict(prefixes=prefixes, drafts=drafts, seed=seed))


def lognormal_prefixes(seed: int, n: int, median: float = 16384.0, sigma: float = 1.0,
                       lo: int = 2048, hi: int = 131072) -> list:
    """ln P ~ N(ln median, sigma^2), clipped to [lo, hi] and rounded to an integer."""
    z = normals(seed, TAG_LEN, n, 1.0)
    p = np.exp(np.log(median) + sigma * z)
    return [int(round(float(min(max(x, lo), hi)))) for x in p]


# The five named workloads (seeded).  Their sizes are those of the target shapes:
#   contiguous_1k   : B=1, P=1024, 16 causal drafts, pool of 1040 rows, identity slots
#   paged_ragged    : B=4, P={4k,8k,16k,32k}, 16 causal drafts, 65,600-slot pool, permuted slots
#   long_185k       : B=1, P=185,000, 16 causal drafts, 200,000-slot pool, permuted slots
#   tree_32k        : B=8, P=32,768, 64-node draft trees (depth <= 8), pool = sum N_b, permuted
#   sweep_q{1,4,16} : B=32, lognormal P (median 16k, clipped 2k..128k), Q in {1,4,16}
#   long_120k       : B=1, P=120,000, 16 causal drafts, 130,000-slot pool (the profiling case: its 150 MB of
#                     KV rows exceed the L2 while the device holds well under 1 GB)
WORKLOADS = ("contiguous_1k", "paged_ragged", "long_185k", "tree_32k", "sweep_q1", "sweep_q4", "sweep_q16",
             "long_120k")


def workload(name: str, num_heads: int = NUM_HEADS) -> Case:
    if name == "contiguous_1k":
        return make_case(name, [1024], 16, num_heads=num_heads, pool_slots=1040, permute=False, seed=1)
    if name == "paged_ragged":
        return make_case(name, [4096, 8192, 16384, 32768], 16, num_heads=num_heads, pool_slots=65600, seed=2)
    if name == "long_185k":
        return make_case(name, [185000], 16, num_heads=num_heads, pool_slots=200000, seed=3)
    if name == "long_120k":
        return make_case(name, [120000], 16, num_heads=num_heads, pool_slots=130000, seed=9)
    if name == "tree_32k":
        return make_case(name, [32768] * 8, 64, num_heads=num_heads, tree_depth=8, seed=4)
    if name.startswith("sweep_q"):
        qd = int(name[len("sweep_q"):])
        prefixes = lognormal_prefixes(5, 32)
        return make_case(name, prefixes, qd, num_heads=num_heads, seed=5)
    raise KeyError(name)


def workload_sizes(name: str) -> dict:
    """Shapes of a named workload without drawing its values (cheap)."""
    if name == "contiguous_1k":
        pre, q = [1024], [16]
    elif name == "paged_ragged":
        pre, q = [4096, 8192, 16384, 32768], [16] * 4
    elif name == "long_185k":
        pre, q = [185000], [16]
    elif name == "long_120k":
        pre, q = [120000], [16]
    elif name == "tree_32k":
        pre, q = [32768] * 8, [64] * 8
    elif name.startswith("sweep_q"):
        pre = lognormal_prefixes(5, 32)
        q = [int(name[len("sweep_q"):])] * 32
    else:
        raise KeyError(name)
    return dict(prefixes=pre, drafts=q)
