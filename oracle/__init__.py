"""CPU fp64 oracle for MLA speculative-decoding verify attention.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg are the only callers.  The product path never imports this
package; it shares no code with the GPU path (only the seeded input generator
is common to both).

The arithmetic lives in verify_oracle.c (plain C, fp64, pthreads over query
rows); this module compiles it with gcc when the shared object is missing or
older than the source, and wraps it for numpy arrays.  See the C file's
header for the definition it evaluates and the passages it follows.

Parity status of each function (what pins it is listed in the tests):
  verify / verify_rows  pinned: library SDPA, closed forms, invariants
  verify_split          pinned: equals the unsplit result (merge identity)
  merge                 pinned: closed forms, equals the unsplit result
  tree_masks            pinned: graph-library ancestor sets
  tree_accept           pinned: hand-worked trees, brute force over all root paths
  e4m3_value /          pinned: torch's float8_e4m3fn for all 256 codes; RNE ties
  dequantize_e4m3
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "verify_oracle.c")
LIB = os.path.join(_HERE, "liboracle.so")
D_QK = 576
D_V = 512

_lib = None


def build(src: str = SRC, out: str = LIB, force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE fp64 throughout)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = f"{out}.{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def _bind(path: str):
    L = ctypes.CDLL(path)
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    prob = [vp, vp, i64, vp, vp, vp, vp, vp, i32, i32, dbl]
    L.oracle_verify.argtypes = prob + [vp, vp, i32]
    L.oracle_verify_rows.argtypes = prob + [vp, i64, vp, vp, i32]
    L.oracle_verify_split.argtypes = prob + [i32, vp, vp, i32]
    L.oracle_merge.argtypes = [vp, vp, i32, i64, i32, vp, vp]
    L.oracle_tree_masks.argtypes = [vp, vp, i32, vp]
    L.oracle_num_cpus.argtypes = []
    for f in (L.oracle_verify, L.oracle_verify_rows, L.oracle_verify_split, L.oracle_merge,
              L.oracle_tree_masks, L.oracle_num_cpus):
        f.restype = ctypes.c_int
    return L


def lib(path: Optional[str] = None):
    """The loaded oracle library (built on first use); `path` loads another build."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        _lib = _bind(build())
    return _lib


def num_cpus() -> int:
    return int(lib().oracle_num_cpus())


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _prob(case, draft_mask: Optional[np.ndarray], use_parent: bool = True):
    q = np.ascontiguousarray(case.q, dtype=np.uint16)
    kv = np.ascontiguousarray(case.kv_pool, dtype=np.uint16)
    kvp = np.ascontiguousarray(case.kv_indptr, dtype=np.int32)
    kvi = np.ascontiguousarray(case.kv_indices, dtype=np.int32)
    qop = np.ascontiguousarray(case.qo_indptr, dtype=np.int32)
    dm = None if draft_mask is None else np.ascontiguousarray(draft_mask, dtype=np.uint64)
    par = None
    if use_parent and case.parent is not None and dm is None:
        par = np.ascontiguousarray(case.parent, dtype=np.int32)
    keep = (q, kv, kvp, kvi, qop, dm, par)
    args = [q.ctypes.data, kv.ctypes.data, kv.shape[0], kvp.ctypes.data, kvi.ctypes.data, qop.ctypes.data,
            _ptr(dm), _ptr(par), len(kvp) - 1, q.shape[1], float(case.sm_scale)]
    return keep, args


def verify(case, draft_mask: Optional[np.ndarray] = None, threads: int = 0, lib_=None):
    """Every row: (out [T_q, H, 512] f64, lse [T_q, H] f64)."""
    L = lib_ or lib()
    keep, args = _prob(case, draft_mask)
    T, H = case.q.shape[0], case.q.shape[1]
    out = np.zeros((T, H, D_V), dtype=np.float64)
    lse = np.zeros((T, H), dtype=np.float64)
    rc = L.oracle_verify(*args, out.ctypes.data, lse.ctypes.data, threads)
    if rc != 0:
        raise ValueError("oracle_verify rejected its inputs")
    return out, lse


def verify_rows(case, rows: np.ndarray, draft_mask: Optional[np.ndarray] = None, threads: int = 0, lib_=None):
    """Selected rows (global id t*H + h): (out [n, 512], lse [n])."""
    L = lib_ or lib()
    keep, args = _prob(case, draft_mask)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), D_V), dtype=np.float64)
    lse = np.zeros(len(rows), dtype=np.float64)
    rc = L.oracle_verify_rows(*args, rows.ctypes.data, len(rows), out.ctypes.data, lse.ctypes.data, threads)
    if rc != 0:
        raise ValueError("oracle_verify_rows rejected its inputs")
    return out, lse


def verify_split(case, splits: int, draft_mask: Optional[np.ndarray] = None, threads: int = 0, lib_=None):
    L = lib_ or lib()
    keep, args = _prob(case, draft_mask)
    T, H = case.q.shape[0], case.q.shape[1]
    out = np.zeros((T, H, D_V), dtype=np.float64)
    lse = np.zeros((T, H), dtype=np.float64)
    rc = L.oracle_verify_split(*args, int(splits), out.ctypes.data, lse.ctypes.data, threads)
    if rc != 0:
        raise ValueError("oracle_verify_split rejected its inputs")
    return out, lse


def merge(o_parts: np.ndarray, lse_parts: np.ndarray, lib_=None):
    """o_parts [S, R, D], lse_parts [S, R] -> (o [R, D], lse [R])."""
    L = lib_ or lib()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, R, D = o_parts.shape
    o = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    L.oracle_merge(o_parts.ctypes.data, lse_parts.ctypes.data, S, R, D, o.ctypes.data, lse.ctypes.data)
    return o, lse


def tree_masks(parent: np.ndarray, qo_indptr: np.ndarray, lib_=None) -> np.ndarray:
    L = lib_ or lib()
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    qo_indptr = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    out = np.zeros(int(qo_indptr[-1]), dtype=np.uint64)
    rc = L.oracle_tree_masks(parent.ctypes.data, qo_indptr.ctypes.data, len(qo_indptr) - 1, out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_tree_masks: parents must precede their children")
    return out


def tree_accept(qo_indptr: np.ndarray, parent: Optional[np.ndarray], draft_token: np.ndarray,
                target_token: np.ndarray, root_token: np.ndarray):
    """Greedy acceptance of a verified draft tree (plain Python; small trees).

    The pages name a tree_accept kernel run after the verify attention but do
    not describe it; this is the plain reading of greedy tree verification.
    Draft node i of a sequence proposes draft_token[i] after its parent (the
    prefix for a root, parent -1); the target's greedy token after node j is
    target_token[j], and after the prefix root_token.  A node is accepted when
    its parent is accepted (the prefix always is) and its token equals the
    target's token after the parent.  The chosen path ends at the deepest
    accepted node (the smallest index among equally deep ones).

    Returns accept_len [B] (nodes on the path), accept_path [T] (each
    sequence's path, root first, from its first position; -1 after it),
    next_token [B] (the target's token after the path's last node, or after
    the prefix) and bad [B] (parents not in [-1, i); nothing accepted).
    parent None means the chain parent[i] = i - 1.
    """
    qo = np.asarray(qo_indptr, np.int64)
    B = len(qo) - 1
    T = int(qo[-1])
    accept_len = np.zeros(B, np.int32)
    accept_path = np.full(T, -1, np.int32)
    next_token = np.zeros(B, np.int32)
    bad = np.zeros(B, bool)
    for b in range(B):
        q0, n = int(qo[b]), int(qo[b + 1] - qo[b])
        par = [int(parent[q0 + i]) if parent is not None else i - 1 for i in range(n)]
        if any(p < -1 or p >= i for i, p in enumerate(par)):
            bad[b] = True
            next_token[b] = root_token[b]
            continue
        accepted = [False] * n
        depth = [0] * n
        best = -1
        for i in range(n):
            p = par[i]
            expected = root_token[b] if p < 0 else target_token[q0 + p]
            accepted[i] = (p < 0 or accepted[p]) and draft_token[q0 + i] == expected
            depth[i] = 0 if p < 0 else depth[p] + 1
            if accepted[i] and (best < 0 or depth[i] > depth[best]):
                best = i
        if best < 0:
            next_token[b] = root_token[b]
            continue
        path = []
        node = best
        while node >= 0:
            path.append(node)
            node = par[node]
        path.reverse()
        accept_len[b] = len(path)
        accept_path[q0:q0 + len(path)] = path
        next_token[b] = target_token[q0 + best]
    return accept_len, accept_path, next_token, bad


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    """Exact value of 8-bit e4m3 codes (OCP FP8 "E4M3": 1 sign, 4 exponent bits
    with bias 7, 3 mantissa bits; exponent field 0 is subnormal, 2^-6 * m/8;
    S.1111.111 is NaN; no infinities), as float64."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mag = np.where((e == 0xF) & (m == 0x7), np.nan, mag)
    return sign * mag


def _bf16_rne_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest, ties to even (finite inputs)."""
    b = np.asarray(x32, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def dequantize_e4m3(codes: np.ndarray, scale: float) -> np.ndarray:
    """An fp8 latent row's bf16 value: the code's value times the pool's scale,
    rounded to float32 and then to bf16 (both round to nearest even), as bf16
    bit patterns.  This is the reading used for fp8 KV storage: the pages do
    not describe one."""
    v32 = e4m3_value(codes).astype(np.float32) * np.float32(scale)
    return _bf16_rne_bits(v32)
