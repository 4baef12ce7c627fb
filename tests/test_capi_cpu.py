"""C-ABI library checks that need no GPU: it loads, exports every declared
symbol, validates arguments before touching a device, and plans splits."""
import ctypes
import os
import re

import numpy as np
import pytest

from speculative_decoding_mla_gb300 import build as vbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    vbuild.build()
    from speculative_decoding_mla_gb300 import binding
    return binding


def declared_functions():
    text = open(os.path.join(ROOT, "include", "verify_attn_mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(verify_attn_mla\w*)\s*\(", text)))


def test_library_exports_every_declared_symbol(B):
    names = declared_functions()
    assert len(names) >= 10
    L = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(B.EXPORTS)


def test_status_strings(B):
    assert B.status_string(0) == "ok"
    for code in range(-9, 0):
        assert B.status_string(code) != "unknown status"
    assert B.verify_attn_mla_version() >= 100


def _run_raw(B, **kw):
    args = dict(q=None, kv=None, S=16, kvp=None, kvi=None, qop=None, dm=None, par=None,
                kvh=np.array([0, 8], np.int32), qoh=np.array([0, 2], np.int32), batch=1, H=4, scale=0.1,
                splits=0, out=None, lse=None, ws=None, wsb=0, stream=None)
    args.update(kw)
    kvh, qoh = args["kvh"], args["qoh"]
    return B.lib().verify_attn_mla(args["q"], args["kv"], args["S"], args["kvp"], args["kvi"], args["qop"],
                                   args["dm"], args["par"], kvh.ctypes.data if kvh is not None else None,
                                   qoh.ctypes.data if qoh is not None else None, args["batch"], args["H"],
                                   args["scale"], args["splits"], args["out"], args["lse"], args["ws"], args["wsb"],
                                   args["stream"])


def test_argument_errors_before_any_launch(B):
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    good = dict(q=fake, kv=fake, kvp=fake, kvi=fake, qop=fake, out=fake, lse=fake, ws=fake * 2, wsb=1 << 20)
    assert _run_raw(B, **{**good, "kvh": None}) == B.VMLA_ERR_NULL
    assert _run_raw(B, **{**good, "ws": None}) == B.VMLA_ERR_NULL
    assert _run_raw(B, **{**good, "q": None}) == B.VMLA_ERR_NULL
    assert _run_raw(B, **{**good, "H": 0}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "batch": -1}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "qoh": np.array([0, 65], np.int32), "kvh": np.array([0, 80], np.int32)}) == \
        B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "qoh": np.array([0, 9], np.int32)}) == B.VMLA_ERR_SHAPE  # drafts > keys
    assert _run_raw(B, **{**good, "kvh": np.array([1, 8], np.int32)}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "splits": 65}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "splits": -2}) == B.VMLA_ERR_SHAPE  # -1 is VMLA_SPLITS_LANES
    assert _run_raw(B, **{**good, "scale": 0.0}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "scale": -0.1}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "scale": float("inf")}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "scale": float("nan")}) == B.VMLA_ERR_SHAPE
    assert _run_raw(B, **{**good, "q": fake + 2}) == B.VMLA_ERR_ALIGN
    assert _run_raw(B, **{**good, "ws": fake + 16}) == B.VMLA_ERR_ALIGN
    # valid arguments on a machine without an sm_103 device
    import torch
    if not torch.cuda.is_available():
        assert _run_raw(B, **good) == B.VMLA_ERR_DEVICE


def _run_dplan(B, fn="verify_attn_mla_device_plan", **kw):
    args = dict(q=None, kv=None, S=16, kvp=None, kvi=None, qop=None, dm=None, par=None, batch=1, H=4, maxq=2,
                maxkv=8, scale=0.1, splits=0, out=None, lse=None, ws=None, wsb=0, stream=None)
    args.update(kw)
    return getattr(B.lib(), fn)(args["q"], args["kv"], args["S"], args["kvp"], args["kvi"],
                                               args["qop"], args["dm"], args["par"], args["batch"], args["H"],
                                               args["maxq"], args["maxkv"], args["scale"], args["splits"],
                                               args["out"], args["lse"], args["ws"], args["wsb"], args["stream"])


def test_device_plan_argument_errors_before_any_launch(B):
    fake = 1 << 20  # never dereferenced: every case below fails validation first
    good = dict(q=fake, kv=fake, kvp=fake, kvi=fake, qop=fake, out=fake, lse=fake, ws=fake * 2, wsb=1 << 20)
    assert _run_dplan(B, **{**good, "ws": None}) == B.VMLA_ERR_NULL
    assert _run_dplan(B, **{**good, "kvp": None}) == B.VMLA_ERR_NULL
    assert _run_dplan(B, **{**good, "q": None}) == B.VMLA_ERR_NULL
    assert _run_dplan(B, **{**good, "batch": -1}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "batch": 513}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "H": 0}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "maxq": 65}) == B.VMLA_ERR_SHAPE  # more than 64 drafts per sequence
    assert _run_dplan(B, **{**good, "maxq": -1}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "maxkv": -1}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "maxkv": 1 << 31}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "splits": 65}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "scale": 0.0}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "scale": float("nan")}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "S": 0}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, **{**good, "q": fake + 2}) == B.VMLA_ERR_ALIGN
    # the same call on pool runs (run_base in kv_indices' place)
    runs = "verify_attn_mla_runs_device_plan"
    assert _run_dplan(B, fn=runs, **{**good, "kvi": None}) == B.VMLA_ERR_NULL  # run_base
    assert _run_dplan(B, fn=runs, **{**good, "kvi": fake + 2}) == B.VMLA_ERR_ALIGN
    assert _run_dplan(B, fn=runs, **{**good, "splits": 65}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, fn=runs, **{**good, "maxq": 65}) == B.VMLA_ERR_SHAPE
    assert _run_dplan(B, fn=runs, **{**good, "ws": None}) == B.VMLA_ERR_NULL
    assert _run_dplan(B, **{**good, "ws": fake + 16}) == B.VMLA_ERR_ALIGN
    import ctypes
    n = ctypes.c_size_t(0)
    assert B.lib().verify_attn_mla_device_plan_workspace_size(1, 64, 16, 1000, 0, None) == B.VMLA_ERR_NULL
    assert B.lib().verify_attn_mla_device_plan_workspace_size(1, 64, 65, 1000, 0, ctypes.byref(n)) == \
        B.VMLA_ERR_SHAPE
    import torch
    if not torch.cuda.is_available():
        assert _run_dplan(B, **good) == B.VMLA_ERR_DEVICE
        assert B.lib().verify_attn_mla_device_plan_workspace_size(1, 64, 16, 1000, 0, ctypes.byref(n)) == \
            B.VMLA_ERR_DEVICE


def test_defrag_and_runs_argument_errors_before_any_launch(B):
    fake = 1 << 20
    L = B.lib()
    kvh = np.array([0, 8], np.int32)
    def defrag(**kw):
        a = dict(src=fake, ss=16, kvp=fake, kvi=fake, kvh=kvh.ctypes.data, batch=1, dst=fake, ds=64, base=fake,
                 st=None, stream=None)
        a.update(kw)
        return L.verify_attn_mla_defrag(*a.values())
    assert defrag(kvh=None) == B.VMLA_ERR_NULL
    assert defrag(batch=-1) == B.VMLA_ERR_SHAPE
    assert defrag(ds=-1) == B.VMLA_ERR_SHAPE
    assert defrag(kvh=np.array([0, -3], np.int32).ctypes.data) == B.VMLA_ERR_SHAPE
    assert defrag(kvh=np.array([2, 8], np.int32).ctypes.data) == B.VMLA_ERR_SHAPE
    assert defrag(dst=None) == B.VMLA_ERR_NULL
    assert defrag(base=None) == B.VMLA_ERR_NULL
    assert defrag(src=fake + 4) == B.VMLA_ERR_ALIGN
    assert defrag(kvh=np.array([0, 0], np.int32).ctypes.data) == B.VMLA_OK  # nothing to copy
    qoh = np.array([0, 2], np.int32)
    def runs(**kw):
        a = dict(q=fake, kv=fake, S=16, kvp=fake, base=fake, qop=fake, dm=None, par=None, kvh=kvh.ctypes.data,
                 qoh=qoh.ctypes.data, batch=1, H=4, scale=0.1, splits=0, out=fake, lse=fake, ws=fake * 2,
                 wsb=1 << 20, stream=None)
        a.update(kw)
        return L.verify_attn_mla_runs(*a.values())
    assert runs(base=None) == B.VMLA_ERR_NULL
    assert runs(kvp=None) == B.VMLA_ERR_NULL
    assert runs(H=0) == B.VMLA_ERR_SHAPE
    assert runs(scale=0.0) == B.VMLA_ERR_SHAPE
    assert runs(base=fake + 2) == B.VMLA_ERR_ALIGN
    def append(**kw):
        a = dict(src=fake, ss=16, kvp=fake, kvi=fake, kvh=kvh.ctypes.data, batch=1, dst=fake, ds=64, base=fake,
                 first=fake, mx=0, st=None, stream=None)
        a.update(kw)
        return L.verify_attn_mla_defrag_append(*a.values())
    assert append(first=None) == B.VMLA_ERR_NULL
    assert append(first=fake + 2) == B.VMLA_ERR_ALIGN
    assert append(batch=-1) == B.VMLA_ERR_SHAPE
    assert append(mx=-1) == B.VMLA_ERR_SHAPE
    assert append(kvh=np.array([0, 0], np.int32).ctypes.data, first=None) == B.VMLA_OK  # nothing to copy
    import torch
    if not torch.cuda.is_available():
        assert defrag() == B.VMLA_ERR_DEVICE
        assert runs() == B.VMLA_ERR_DEVICE
        assert append() == B.VMLA_ERR_DEVICE


def test_fp8_argument_errors_before_any_launch(B):
    fake = 1 << 20
    L = B.lib()
    kvh, qoh = np.array([0, 8], np.int32), np.array([0, 2], np.int32)
    def call(scale=0.05, **kw):
        a = dict(q=fake, kv=fake, S=16, scale=scale, kvp=fake, kvi=fake, qop=fake, dm=None, par=None,
                 kvh=kvh.ctypes.data, qoh=qoh.ctypes.data, batch=1, H=4, sm=0.1, splits=0, out=fake, lse=fake,
                 ws=fake * 2, wsb=1 << 20, stream=None)
        a.update(kw)
        return L.verify_attn_mla_fp8(*a.values())
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert call(scale=bad) == B.VMLA_ERR_SHAPE
    assert call(kvi=None) == B.VMLA_ERR_NULL
    assert call(q=fake + 2) == B.VMLA_ERR_ALIGN
    import torch
    if not torch.cuda.is_available():
        assert call() == B.VMLA_ERR_DEVICE


def test_test_fault_hook_arguments(B):
    L = B.lib()
    assert L.verify_attn_mla_test_fault(2, 0) == B.VMLA_ERR_SHAPE
    assert L.verify_attn_mla_test_fault(0, -1) == B.VMLA_ERR_SHAPE
    assert L.verify_attn_mla_test_fault(1, 1000) == B.VMLA_OK
    assert L.verify_attn_mla_test_fault(0, 0) == B.VMLA_OK


def test_tree_accept_argument_errors_before_any_launch(B):
    fake = 1 << 20
    L = B.lib()
    good = [fake, fake, fake, fake, fake, 2, 10, fake, fake, fake, None, None]
    def call(i=None, v=None):
        a = list(good)
        if i is not None:
            a[i] = v
        return L.verify_attn_mla_tree_accept(*a)
    assert call(5, -1) == B.VMLA_ERR_SHAPE
    assert call(6, 129) == B.VMLA_ERR_SHAPE  # more than 64 nodes per sequence
    assert call(6, -1) == B.VMLA_ERR_SHAPE
    assert call(0, None) == B.VMLA_ERR_NULL
    assert call(4, None) == B.VMLA_ERR_NULL
    assert call(2, None) == B.VMLA_ERR_NULL
    assert call(8, None) == B.VMLA_ERR_NULL
    assert call(2, fake + 2) == B.VMLA_ERR_ALIGN
    assert L.verify_attn_mla_tree_accept(None, None, None, None, None, 0, 0, None, None, None, None, None) == B.VMLA_OK
    import torch
    if not torch.cuda.is_available():
        assert call() == B.VMLA_ERR_DEVICE


def _plan(B, kernel, prefixes, drafts, H=64, splits=0, sms=152):
    qo = np.zeros(len(prefixes) + 1, np.int32)
    qo[1:] = np.cumsum(drafts)
    kv = np.zeros(len(prefixes) + 1, np.int32)
    kv[1:] = np.cumsum(np.array(prefixes) + np.array(drafts))
    info, per = B.verify_attn_mla_plan(kernel, qo, kv, H, splits, sms)
    return info, per, qo, kv


@pytest.mark.parametrize("kernel", [0, 1])
def test_plan_covers_work(B, kernel):
    rpu = 256 if kernel == 0 else 32
    for prefixes, drafts in [([185000], [16]), ([4096, 8192, 16384, 32768], [16] * 4), ([1024], [16]),
                             ([32768] * 8, [64] * 8), ([3, 0, 70000], [1, 0, 4])]:
        info, per, qo, kv = _plan(B, kernel, prefixes, drafts)
        units = 0
        part = 0
        merge = 0
        for b in range(len(prefixes)):
            nq, nk = drafts[b], prefixes[b] + drafts[b]
            if nq == 0:
                continue
            rows = nq * 64
            s = int(per[b])
            assert 1 <= s <= 64
            assert s <= max(1, nk)
            units += -(-rows // rpu) * s
            if s > 1:
                part += rows * s
                merge += rows
        assert info.num_units == units
        assert info.partial_rows == part and info.merge_rows == merge
        assert info.workspace_bytes >= part * 512 * 4


def test_plan_fills_the_gpu_for_one_long_sequence(B):
    info, per, _, _ = _plan(B, 0, [185000], [16])
    # 4 row blocks of 256 rows on 38 four-SM clusters: several key pieces each
    assert per[0] >= 8 and info.num_units >= 64
    info, per, _, _ = _plan(B, 0, [185000], [16], splits=3)
    assert per[0] == 3 and info.num_units == 12


def test_plan_accepts_more_units_than_one_launch(B):
    # 16 x 4 row pairs x 64 forced pieces: more units than one tensor-core launch schedules
    info, per, _, _ = _plan(B, 0, [8176] * 16, [16] * 16, splits=64)
    assert info.num_units == 4096 and all(int(p) == 64 for p in per)
    # the largest shapes the header allows plan on both kernels
    for kernel in (0, 1):
        info, per, _, _ = _plan(B, kernel, [2000] * 512, [64] * 512, H=128)
        assert info.num_units > 0


def test_plan_rejects_bad_shapes(B):
    with pytest.raises(B.VmlaError):
        _plan(B, 0, [10], [65])
    with pytest.raises(B.VmlaError):
        B.verify_attn_mla_plan(0, np.array([0, 4], np.int32), np.array([0, 2], np.int32), 64)


def test_plan_units_within_the_device_plan_bound(B):
    """The device-planned call sizes its partial area for caller bounds before any length is known:
    with C clusters the automatic plan makes at most 12C units (its largest candidate aims at 12
    units per cluster) plus one per row block, each of 256 rows, and never more than 64 pieces of
    every query row; a lane plan makes at most C + 2 per row block (a stream of T tiles meets at most
    (T - 1) / L + 2 lanes).  The host planner runs the same split arithmetic; check that bound on
    random length sets."""
    rng = np.random.default_rng(7)
    for trial in range(300):
        batch = int(rng.integers(1, 40))
        H = int(rng.choice([8, 16, 64, 128]))
        drafts = rng.integers(0, 65, batch)
        prefixes = np.where(rng.random(batch) < 0.5, rng.integers(0, 3000, batch), rng.integers(0, 200000, batch))
        clusters = int(rng.integers(1, 40))
        info, per, qo, kv = _plan(B, 0, prefixes.tolist(), drafts.tolist(), H=H, sms=4 * clusters)
        rows = int(qo[-1]) * H
        row_blocks = -(-rows // 256) + batch
        cap = min(256 * (12 * clusters + 2 * row_blocks), rows * 64)
        assert info.num_units <= 12 * clusters + 2 * row_blocks
        assert info.partial_rows <= cap
        if info.lane_width:
            assert info.num_units <= clusters + 2 * row_blocks
    # forced piece counts: at most `splits` pieces of every row block
    for splits in (1, 3, 17, 64):
        info, per, qo, kv = _plan(B, 0, [5000, 100, 70000], [16, 3, 64], H=64, splits=splits, sms=144)
        row_blocks = -(-int(qo[-1]) * 64 // 256) + 3
        assert info.num_units <= splits * row_blocks
        assert info.partial_rows <= min(256 * splits * row_blocks, int(qo[-1]) * 64 * 64)


def test_binding_checks_array_arguments_before_the_call(B):
    """The binding refuses, before calling the library, arrays the C ABI cannot check from a bare
    pointer: host memory where device memory is read, the wrong element size, strided views."""
    import torch
    T, H, N = 2, 8, 40
    kvp = np.array([0, N], np.int32)
    qop = np.array([0, T], np.int32)
    kv = torch.zeros((N, 576), dtype=torch.bfloat16)
    kvi = torch.arange(N, dtype=torch.int32)
    out = torch.zeros((T, H, 512), dtype=torch.bfloat16)
    lse = torch.zeros((T, H), dtype=torch.float32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)

    def call(q):
        B.verify_attn_mla(q, kv, torch.from_numpy(kvp), kvi, torch.from_numpy(qop), kvp, qop, out, lse, ws, 0.07)

    # through an entry point (its first array argument is checked first)
    with pytest.raises(ValueError, match="q: device memory expected, got cpu"):
        call(torch.zeros((T, H, 576), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="q: device memory expected, got a numpy array"):
        call(np.zeros((T, H, 576), np.uint16))
    with pytest.raises(ValueError, match="q: 2-byte elements expected"):
        call(torch.zeros((T, H, 576), dtype=torch.float32))
    with pytest.raises(ValueError, match="q_host: 2-byte elements expected"):
        B.verify_attn_mla_host(torch.zeros((T, H, 576), dtype=torch.float32), kv, kvp, kvi, qop, out, lse, ws, 0.07)
    # each rule of the check
    with pytest.raises(ValueError, match="kv_pool: not contiguous"):
        B._arg(torch.zeros((576, N), dtype=torch.bfloat16).t(), 2, "kv_pool", False)
    with pytest.raises(ValueError, match="kv_indices: not contiguous"):
        B._arg(np.zeros((8, 2), np.int32)[:, 0], 4, "kv_indices", False)
    with pytest.raises(ValueError, match="kv_indices: 4-byte elements expected"):
        B._arg(torch.zeros(4, dtype=torch.int64), 4, "kv_indices", False)
    assert B._arg(None, 4, "parent", True) is None
    a = np.zeros(3, np.int32)
    assert B._arg(a, 4, "kv_indices_host", False) == a.ctypes.data
    t = torch.zeros(5, dtype=torch.uint8)
    assert B._arg(t, 0, "workspace", False) == t.data_ptr()


def test_prepared_call_marshals_once_and_reports_errors(B):
    # a prepared call converts its arguments to the entry point's C types once and repeats the call
    ok = B.Prepared(B.lib().verify_attn_mla_test_fault, "verify_attn_mla_test_fault", (0, 0), ())
    ok()
    ok()
    bad = B.Prepared(B.lib().verify_attn_mla_test_fault, "verify_attn_mla_test_fault", (5, 0), ())
    with pytest.raises(B.VmlaError) as e:
        bad()
    assert e.value.status == B.VMLA_ERR_SHAPE


def _piece_rule(qo, kv, H, clusters, search=True):
    """The tensor-core planner's piece-size rule, stated on its own: candidate k aims at m_k / 16
    units per cluster (chunk target ceil(16 W / (C m_k)), at least one 128-key tile); a sequence of
    N keys gets ceil(N / target) pieces (at most 64), of a length rounded up to 128 keys; a unit
    costs its keys plus 384; a candidate's score is the longest cluster load when its units, sorted
    by cost (longest first), are dealt to the clusters in a snake order, plus a twentieth of a key
    per fp32 partial row (query rows x pieces of every split sequence) and 128 keys when there is
    any; the best-scoring candidate
    replaces the default (m = 32) only when it scores at least 3 % lower; more than 64 sequences,
    or more than 3072 units, leave the candidate set.

    Then the lane plan (only when the search ran): G = the largest of 4, 3, 2 dividing every
    sequence's row-block count (else 1), C // G lanes (1 to 64 of them); each sequence has
    rb / G streams, each taking ceil(N / 128) tiles and then 5 more in a line of cost W; lanes
    of L = ceil(W / lanes) cut that line, and a stream's pieces are the lanes its tiles meet; a
    sequence's count is the most of any of its streams; the lane plan scores (L + 3) * 128 plus
    the same merge charge and replaces the uniform choice when it scores at least 3 % lower.
    A lane plan's merge rows are the rows of its streams cut into more than one piece.
    Returns the counts and the lane plan's merge rows (None: the uniform plan)."""
    ms = [12 + 2 * k for k in range(10)] + [32 + 4 * k for k in range(10)] + \
         [72 + 8 * k for k in range(8)] + [144 + 16 * k for k in range(4)]
    B = len(qo) - 1
    nq = [int(qo[b + 1] - qo[b]) for b in range(B)]
    nk = [int(kv[b + 1] - kv[b]) for b in range(B)]
    rb = [-(-q * H // 256) for q in nq]
    W = sum(r * n for r, n, q in zip(rb, nk, nq) if q)

    def pieces(target):
        out = []
        for q, n in zip(nq, nk):
            if q == 0:
                out.append((1, max(n, 1)))
                continue
            p = min(max(-(-n // target), 1), 64)
            ch = -(-(-(-n // p)) // 128) * 128
            out.append((-(-n // ch), ch))
        return out

    def target(m):
        return max(128, -(-max(W, 1) * 16 // (clusters * m)))

    def score(m):
        costs = []
        part = 0
        for (p, ch), q, r, n in zip(pieces(target(m)), nq, rb, nk):
            if q == 0:
                continue
            for s in range(p):
                costs += [min(ch, n - s * ch) + 384] * r
            if p > 1:
                part += q * H * p
        if len(costs) > 3072:
            return None
        load = [0] * clusters
        for i, c in enumerate(sorted(costs, reverse=True)):
            rnd, j = divmod(i, clusters)
            load[clusters - 1 - j if rnd % 2 else j] += c
        return max(load) + part // 20 + (128 if part else 0)

    def lanes_plan(uniform_score):
        rbs = [r for r, q in zip(rb, nq) if q]
        G = next((g for g in (4, 3, 2) if all(r % g == 0 for r in rbs)), 1)
        lanes = clusters // G
        if not 1 <= lanes <= 64:
            return None
        W = sum(r // G * (-(-n // 128) + 5) for r, n, q in zip(rb, nk, nq) if q)
        if W < 1:
            return None
        L = max(1, -(-W // lanes))
        pos, counts, part, merge = 0, [], 0, 0
        for r, n, q in zip(rb, nk, nq):
            if q == 0:
                counts.append(1)
                continue
            T = -(-n // 128)
            most = 1
            for g in range(r // G):
                p = (pos + T - 1) // L - pos // L + 1
                most = max(most, p)
                if p > 1:  # the merge combines the rows of this stream's G row blocks
                    merge += min(q * H, (g + 1) * G * 256) - g * G * 256
                pos += T + 5
            counts.append(most)
            if most > 1:
                part += q * H * most
        lane_score = (L + 3) * 128 + part // 20 + (128 if part else 0)
        ok = uniform_score is None or lane_score * 100 < uniform_score * 97
        return (counts, merge) if ok else None

    m_def = 32
    if search and B <= 64:
        scores = [(score(m), k) for k, m in enumerate(ms)]
        valid = [(s, k) for s, k in scores if s is not None]
        d = scores[ms.index(m_def)][0]
        chosen, chosen_score = m_def, d
        if valid:
            s_best, k_best = min(valid)
            if d is None or s_best * 100 < d * 97:
                chosen, chosen_score = ms[k_best], s_best
        if chosen_score is not None:
            lane = lanes_plan(chosen_score)
            if lane is not None:
                return lane[0], lane[1]
        return [p for p, _ in pieces(target(chosen))], None
    return [p for p, _ in pieces(target(m_def))], None


def test_tc_piece_size_rule(B):
    """The host planner's per-sequence piece counts equal the rule stated independently above, on
    the ragged workload shapes and random length sets (the device planner runs the same integer
    arithmetic; its plans are compared bit for bit with the host's on the GPU)."""
    rng = np.random.default_rng(13)
    shapes = [([4096, 8192, 16384, 32768], [16] * 4, 64, 36), ([185000], [16], 64, 36),
              ([32768] * 8, [64] * 8, 64, 36), ([1024], [16], 64, 36)]
    for t in range(120):
        b = int(rng.integers(1, 70))
        prefixes = np.where(rng.random(b) < 0.3, rng.integers(0, 3000, b), rng.integers(0, 120000, b)).tolist()
        drafts = rng.integers(0, 65, b).tolist()
        shapes.append((prefixes, drafts, int(rng.choice([8, 16, 64, 128])), int(rng.integers(1, 40))))
    lane_plans = 0
    for prefixes, drafts, H, clusters in shapes:
        info, per, qo, kv = _plan(B, 0, prefixes, drafts, H=H, sms=4 * clusters)
        want, lane_merge = _piece_rule(qo, kv, H, clusters)
        got = [int(p) for p in per]
        assert (info.lane_width > 0) == (lane_merge is not None), (prefixes, drafts, H, clusters)
        if lane_merge is not None:
            assert info.merge_rows == lane_merge
            lane_plans += 1
        for b in range(len(drafts)):
            if drafts[b] > 0:
                assert got[b] == want[b], (prefixes, drafts, H, clusters, b)
    assert 10 < lane_plans < len(shapes) - 10  # both forms occur
    # the ragged four-sequence batch takes the lane plan: lanes of four clusters (four row blocks per
    # sequence), streams of 33, 65, 129 and 257 tiles cut every 56 cost units into 1, 2, 4 and 5 pieces
    info, per, qo, kv = _plan(B, 0, [4096, 8192, 16384, 32768], [16] * 4, H=64, sms=144)
    assert info.lane_width == 4 and info.lane_count == 9
    assert [int(p) for p in per] == [1, 2, 4, 5]
    assert [int(p) for p in per] != _piece_rule(qo, kv, 64, 36, search=False)[0]
    # one long sequence keeps its equal pieces (one per cluster already balances it)
    info, per, qo, kv = _plan(B, 0, [185000], [16], H=64, sms=144)
    assert info.lane_width == 0 and int(per[0]) == 9
    # VMLA_SPLITS_LANES takes the lane plan wherever it fits (the rule above without the score
    # comparison), also past 64 sequences
    for prefixes, drafts, H, clusters in shapes[:40] + [([700] * 80, [3] * 80, 64, 36)]:
        info, per, qo, kv = _plan(B, 0, prefixes, drafts, H=H, splits=B.VMLA_SPLITS_LANES, sms=4 * clusters)
        rbs = [-(-d * H // 256) for d in drafts if d > 0]
        G = next((g for g in (4, 3, 2) if all(r % g == 0 for r in rbs)), 1)
        assert info.lane_width == (G if 1 <= clusters // G <= 64 and rbs else 0), (prefixes, drafts, H, clusters)
    # the CUDA-core kernel takes it as 0
    i0, p0, _, _ = _plan(B, 1, [5000, 300], [4, 16], H=64)
    i1, p1, _, _ = _plan(B, 1, [5000, 300], [4, 16], H=64, splits=B.VMLA_SPLITS_LANES)
    assert list(p0) == list(p1) and i1.lane_width == 0
