"""Thin Python binding of the C ABI in include/verify_attn_mla.h.

Argument marshalling only: every step of the computation runs in the CUDA
library.  The functions keep the C names and take torch tensors for device
(and pinned host) buffers; `stream` defaults to torch's current stream.  A
status other than VMLA_OK raises VmlaError.  If libvmla.so is missing the
import of this module fails: there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvmla.so")

VMLA_OK = 0
VMLA_ERR_NULL = -1
VMLA_ERR_SHAPE = -2
VMLA_ERR_ALIGN = -3
VMLA_ERR_WORKSPACE = -4
VMLA_ERR_CUDA = -5
VMLA_ERR_TIMEOUT = -6
VMLA_ERR_INDEX = -7
VMLA_ERR_DEVICE = -8
VMLA_ERR_PARENT = -9
VMLA_KERNEL_TC = 0
VMLA_KERNEL_SIMT = 1
VMLA_SPLITS_LANES = -1  # splits value: the tensor-core planner takes its lane plan where it fits
D_QK = 576
D_V = 512

EXPORTS = (
    "verify_attn_mla_plan", "verify_attn_mla_workspace_size", "verify_attn_mla", "verify_attn_mla_simt",
    "verify_attn_mla_merge", "verify_attn_mla_tree_mask", "verify_attn_mla_check",
    "verify_attn_mla_host_buffer_size", "verify_attn_mla_host", "verify_attn_mla_status_string",
    "verify_attn_mla_version", "verify_attn_mla_timing_enable", "verify_attn_mla_timing_read",
    "verify_attn_mla_simt_static", "verify_attn_mla_device_plan_workspace_size", "verify_attn_mla_device_plan",
    "verify_attn_mla_tree_accept", "verify_attn_mla_defrag", "verify_attn_mla_runs",
    "verify_attn_mla_runs_workspace_size", "verify_attn_mla_test_fault", "verify_attn_mla_fp8",
    "verify_attn_mla_simt_static_check", "verify_attn_mla_defrag_append",
    "verify_attn_mla_runs_device_plan_workspace_size", "verify_attn_mla_runs_device_plan",
)


class VmlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_units", ctypes.c_int32), ("max_splits", ctypes.c_int32), ("partial_rows", ctypes.c_int64),
                ("merge_rows", ctypes.c_int64), ("workspace_bytes", ctypes.c_size_t), ("lane_width", ctypes.c_int32),
                ("lane_count", ctypes.c_int32)]


def _load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with speculative_decoding_mla_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    run = [vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp, vp, vp, sz, vp]
    sig = {
        "verify_attn_mla_plan": [i32, i32, i32, vp, vp, i32, i32, ctypes.POINTER(PlanInfo), vp],
        "verify_attn_mla_workspace_size": [i32, i32, vp, vp, i32, ctypes.POINTER(sz)],
        "verify_attn_mla": run,
        "verify_attn_mla_simt": run,
        "verify_attn_mla_merge": [vp, vp, i32, i64, vp, vp, vp],
        "verify_attn_mla_tree_mask": [vp, vp, i32, i32, vp, vp, vp],
        "verify_attn_mla_check": [vp, vp],
        "verify_attn_mla_host_buffer_size": [i32, i32, vp, vp, i32, i32, i32, ctypes.POINTER(sz)],
        "verify_attn_mla_host": [vp, vp, i64, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp, vp, vp, sz, vp],
        "verify_attn_mla_status_string": [i32],
        "verify_attn_mla_version": [],
        "verify_attn_mla_timing_enable": [i32],
        "verify_attn_mla_timing_read": [vp, vp, vp, i32, ctypes.POINTER(i32)],
        "verify_attn_mla_simt_static": [vp, vp, i64, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp, vp, vp],
        "verify_attn_mla_simt_static_check": [vp],
        "verify_attn_mla_device_plan_workspace_size": [i32, i32, i64, i64, i32, ctypes.POINTER(sz)],
        "verify_attn_mla_device_plan": [vp, vp, i64, vp, vp, vp, vp, vp, i32, i32, i64, i64, f32, i32, vp, vp, vp,
                                        sz, vp],
        "verify_attn_mla_runs_device_plan_workspace_size": [i32, i32, i64, i64, i32, ctypes.POINTER(sz)],
        "verify_attn_mla_runs_device_plan": [vp, vp, i64, vp, vp, vp, vp, vp, i32, i32, i64, i64, f32, i32, vp, vp,
                                             vp, sz, vp],
        "verify_attn_mla_tree_accept": [vp, vp, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp],
        "verify_attn_mla_defrag": [vp, i64, vp, vp, vp, i32, vp, i64, vp, vp, vp],
        "verify_attn_mla_defrag_append": [vp, i64, vp, vp, vp, i32, vp, i64, vp, vp, i64, vp, vp],
        "verify_attn_mla_runs": run,
        "verify_attn_mla_runs_workspace_size": [i32, i32, vp, vp, i32, ctypes.POINTER(sz)],
        "verify_attn_mla_test_fault": [i32, i64],
        "verify_attn_mla_fp8": [vp, vp, i64, f32, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp, vp, vp, sz, vp],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_char_p if name == "verify_attn_mla_status_string" else ctypes.c_int
    return L


_lib = _load()


def lib():
    return _lib


def status_string(status: int) -> str:
    return _lib.verify_attn_mla_status_string(int(status)).decode()


def _check(rc: int, where: str):
    if rc != VMLA_OK:
        raise VmlaError(rc, where)


def _arg(t, itemsize: int, name: str, on_device: bool) -> Optional[int]:
    """Pointer of an array argument after the checks the C ABI cannot make from a bare pointer:
    contiguous storage, the element size of the type the entry point reads (0: any) and device or
    host memory as the entry point expects.  Raises ValueError before any call."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        if on_device:
            raise ValueError(f"{name}: device memory expected, got a numpy array")
        if not t.flags.c_contiguous:
            raise ValueError(f"{name}: not contiguous")
        if itemsize and t.itemsize != itemsize:
            raise ValueError(f"{name}: {itemsize}-byte elements expected, got {t.dtype}")
        return t.ctypes.data
    if not t.is_contiguous():
        raise ValueError(f"{name}: not contiguous")
    if itemsize and t.element_size() != itemsize:
        raise ValueError(f"{name}: {itemsize}-byte elements expected, got {t.dtype}")
    if bool(t.is_cuda) != on_device:
        raise ValueError(f"{name}: {'device' if on_device else 'host'} memory expected, got {t.device}")
    return t.data_ptr()


def _d(t, itemsize: int, name: str) -> Optional[int]:
    return _arg(t, itemsize, name, True)


def _h(t, itemsize: int, name: str) -> Optional[int]:
    return _arg(t, itemsize, name, False)


def _host_i32(a) -> np.ndarray:
    if hasattr(a, "cpu"):
        a = a.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def verify_attn_mla_plan(kernel: int, qo_indptr_host, kv_indptr_host, num_heads: int, splits: int = 0,
                         num_sms: int = 152):
    """Host-only split plan: (PlanInfo, splits per sequence)."""
    qo = _host_i32(qo_indptr_host)
    kv = _host_i32(kv_indptr_host)
    B = len(qo) - 1
    info = PlanInfo()
    per = np.zeros(max(B, 1), dtype=np.int32)
    _check(_lib.verify_attn_mla_plan(kernel, B, num_heads, qo.ctypes.data, kv.ctypes.data, splits, num_sms,
                                     ctypes.byref(info), per.ctypes.data), "verify_attn_mla_plan")
    return info, per[:B]


def verify_attn_mla_workspace_size(qo_indptr_host, kv_indptr_host, num_heads: int, splits: int = 0) -> int:
    qo = _host_i32(qo_indptr_host)
    kv = _host_i32(kv_indptr_host)
    n = ctypes.c_size_t(0)
    _check(_lib.verify_attn_mla_workspace_size(len(qo) - 1, num_heads, qo.ctypes.data, kv.ctypes.data, splits,
                                               ctypes.byref(n)), "verify_attn_mla_workspace_size")
    return int(n.value)


class Prepared:
    """One entry-point call whose arguments were checked and marshalled once.  Calling it repeats
    the C call on the same buffers: their contents (and the host indptr arrays' contents) may change
    between calls, their shapes and addresses may not.  It keeps a reference to every array it was
    built from.  Per call this saves the Python checks (about 20 us on the GPU host), which would
    otherwise delay the first kernel of a call made from an idle GPU."""

    __slots__ = ("_fn", "_name", "_args", "_keep")

    def __init__(self, fn, name: str, args, keep):
        self._fn = fn
        self._name = name
        self._args = tuple(t(v) for t, v in zip(fn.argtypes, args))
        self._keep = keep

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != VMLA_OK:
            raise VmlaError(rc, self._name)


def _run_args(q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse, workspace,
              sm_scale, draft_mask=None, parent=None, splits=0, stream=None, num_heads=None, pool_slots=None):
    kvh = _host_i32(kv_indptr_host)
    qoh = _host_i32(qo_indptr_host)
    H = int(num_heads if num_heads is not None else q.shape[1])
    S = int(pool_slots if pool_slots is not None else kv_pool.shape[0])
    args = (_d(q, 2, "q"), _d(kv_pool, 2, "kv_pool"), S, _d(kv_indptr, 4, "kv_indptr"),
            _d(kv_indices, 4, "kv_indices"), _d(qo_indptr, 4, "qo_indptr"), _d(draft_mask, 8, "draft_mask"),
            _d(parent, 4, "parent"), kvh.ctypes.data, qoh.ctypes.data, len(kvh) - 1, H, float(sm_scale), int(splits),
            _d(out, 2, "out"), _d(lse, 4, "lse"), _d(workspace, 0, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream))
    return args, (q, kv_pool, kv_indptr, kv_indices, qo_indptr, kvh, qoh, out, lse, workspace, draft_mask, parent)


def _run(fn, name, *a, **k):
    args, _ = _run_args(*a, **k)
    _check(fn(*args), name)


def prepare_verify_attn_mla(q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
                            workspace, sm_scale, draft_mask=None, parent=None, splits=0, stream=None,
                            kernel: str = "tc") -> Prepared:
    """verify_attn_mla (kernel "tc") or verify_attn_mla_simt ("simt") with its arguments checked and
    marshalled once; call the result to run it."""
    name = "verify_attn_mla" if kernel == "tc" else "verify_attn_mla_simt"
    args, keep = _run_args(q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
                           workspace, sm_scale, draft_mask, parent, splits, stream)
    return Prepared(getattr(_lib, name), name, args, keep)


def verify_attn_mla(q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
                    workspace, sm_scale, draft_mask=None, parent=None, splits=0, stream=None):
    """Tensor-core verify attention into `out` [T,H,512] bf16 and `lse` [T,H] fp32."""
    _run(_lib.verify_attn_mla, "verify_attn_mla", q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host,
         qo_indptr_host, out, lse, workspace, sm_scale, draft_mask, parent, splits, stream)


def _dplan_ws(fn, name, batch, num_heads, max_total_q, max_total_kv, splits):
    n = ctypes.c_size_t(0)
    _check(fn(int(batch), int(num_heads), int(max_total_q), int(max_total_kv), int(splits), ctypes.byref(n)), name)
    return int(n.value)


def verify_attn_mla_device_plan_workspace_size(batch: int, num_heads: int, max_total_q: int, max_total_kv: int,
                                               splits: int = 0) -> int:
    return _dplan_ws(_lib.verify_attn_mla_device_plan_workspace_size, "verify_attn_mla_device_plan_workspace_size",
                     batch, num_heads, max_total_q, max_total_kv, splits)


def verify_attn_mla_runs_device_plan_workspace_size(batch: int, num_heads: int, max_total_q: int, max_total_kv: int,
                                                    splits: int = 0) -> int:
    return _dplan_ws(_lib.verify_attn_mla_runs_device_plan_workspace_size,
                     "verify_attn_mla_runs_device_plan_workspace_size", batch, num_heads, max_total_q, max_total_kv,
                     splits)


def _dplan_call(fn, name, q, kv_pool, kv_indptr, rows, rows_name, qo_indptr, batch, max_total_q, max_total_kv, out,
                lse, workspace, sm_scale, draft_mask, parent, splits, stream, num_heads, pool_slots):
    H = int(num_heads if num_heads is not None else q.shape[1])
    S = int(pool_slots if pool_slots is not None else kv_pool.shape[0])
    rc = fn(_d(q, 2, "q"), _d(kv_pool, 2, "kv_pool"), S, _d(kv_indptr, 4, "kv_indptr"), _d(rows, 4, rows_name),
            _d(qo_indptr, 4, "qo_indptr"), _d(draft_mask, 8, "draft_mask"), _d(parent, 4, "parent"), int(batch), H,
            int(max_total_q), int(max_total_kv), float(sm_scale), int(splits), _d(out, 2, "out"), _d(lse, 4, "lse"),
            _d(workspace, 0, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, name)


def verify_attn_mla_device_plan(q, kv_pool, kv_indptr, kv_indices, qo_indptr, batch: int, max_total_q: int,
                                max_total_kv: int, out, lse, workspace, sm_scale, draft_mask=None, parent=None,
                                splits=0, stream=None, num_heads=None, pool_slots=None):
    """Stream-capture-safe verify attention: the plan is built on the device from the device indptr arrays."""
    _dplan_call(_lib.verify_attn_mla_device_plan, "verify_attn_mla_device_plan", q, kv_pool, kv_indptr, kv_indices,
                "kv_indices", qo_indptr, batch, max_total_q, max_total_kv, out, lse, workspace, sm_scale, draft_mask,
                parent, splits, stream, num_heads, pool_slots)


def verify_attn_mla_runs_device_plan(q, kv_pool, kv_indptr, run_base, qo_indptr, batch: int, max_total_q: int,
                                     max_total_kv: int, out, lse, workspace, sm_scale, draft_mask=None, parent=None,
                                     splits=0, stream=None, num_heads=None, pool_slots=None):
    """verify_attn_mla_runs with the plan built on the device (capture-safe; rows read from their pool runs)."""
    _dplan_call(_lib.verify_attn_mla_runs_device_plan, "verify_attn_mla_runs_device_plan", q, kv_pool, kv_indptr,
                run_base, "run_base", qo_indptr, batch, max_total_q, max_total_kv, out, lse, workspace, sm_scale,
                draft_mask, parent, splits, stream, num_heads, pool_slots)


def verify_attn_mla_defrag(src_pool, kv_indptr, kv_indices, kv_indptr_host, dst_pool, run_base, status_word=None,
                           stream=None):
    """Copies every sequence's rows into its run of dst_pool (runs start at run_base) and zeroes each run's tail."""
    kvh = _host_i32(kv_indptr_host)
    rc = _lib.verify_attn_mla_defrag(_d(src_pool, 2, "src_pool"), int(src_pool.shape[0]),
                                     _d(kv_indptr, 4, "kv_indptr"), _d(kv_indices, 4, "kv_indices"),
                                     kvh.ctypes.data, len(kvh) - 1, _d(dst_pool, 2, "dst_pool"),
                                     int(dst_pool.shape[0]), _d(run_base, 4, "run_base"),
                                     _d(status_word, 4, "status_word"), _stream(stream))
    _check(rc, "verify_attn_mla_defrag")


def _append_args(src_pool, kv_indptr, kv_indices, kv_indptr_host, dst_pool, run_base, first_row, status_word=None,
                 stream=None, max_new_rows=0):
    kvh = _host_i32(kv_indptr_host)
    args = (_d(src_pool, 2, "src_pool"), int(src_pool.shape[0]), _d(kv_indptr, 4, "kv_indptr"),
            _d(kv_indices, 4, "kv_indices"), kvh.ctypes.data, len(kvh) - 1, _d(dst_pool, 2, "dst_pool"),
            int(dst_pool.shape[0]), _d(run_base, 4, "run_base"), _d(first_row, 4, "first_row"), int(max_new_rows),
            _d(status_word, 4, "status_word"), _stream(stream))
    return args, (src_pool, kv_indptr, kv_indices, kvh, dst_pool, run_base, first_row, status_word)


def verify_attn_mla_defrag_append(src_pool, kv_indptr, kv_indices, kv_indptr_host, dst_pool, run_base, first_row,
                                  status_word=None, stream=None, max_new_rows=0):
    """The defragmentation for a decode loop: rows below first_row[b] are already in sequence b's run
    (max_new_rows: a bound on the new rows per sequence, or 0)."""
    args, _ = _append_args(src_pool, kv_indptr, kv_indices, kv_indptr_host, dst_pool, run_base, first_row,
                           status_word, stream, max_new_rows)
    _check(_lib.verify_attn_mla_defrag_append(*args), "verify_attn_mla_defrag_append")


def prepare_verify_attn_mla_defrag_append(*a, **k) -> Prepared:
    """verify_attn_mla_defrag_append with its arguments checked and marshalled once."""
    args, keep = _append_args(*a, **k)
    return Prepared(_lib.verify_attn_mla_defrag_append, "verify_attn_mla_defrag_append", args, keep)


def verify_attn_mla_runs_workspace_size(qo_indptr_host, kv_indptr_host, num_heads: int, splits: int = 0) -> int:
    qo = _host_i32(qo_indptr_host)
    kv = _host_i32(kv_indptr_host)
    n = ctypes.c_size_t(0)
    _check(_lib.verify_attn_mla_runs_workspace_size(len(qo) - 1, num_heads, qo.ctypes.data, kv.ctypes.data, splits,
                                                    ctypes.byref(n)), "verify_attn_mla_runs_workspace_size")
    return int(n.value)


def verify_attn_mla_runs(q, kv_pool, kv_indptr, run_base, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
                         workspace, sm_scale, draft_mask=None, parent=None, splits=0, stream=None):
    """Tensor-core verify attention on rows that lie in per-sequence runs of the pool (no gather)."""
    _run(_lib.verify_attn_mla_runs, "verify_attn_mla_runs", q, kv_pool, kv_indptr, run_base, qo_indptr,
         kv_indptr_host, qo_indptr_host, out, lse, workspace, sm_scale, draft_mask, parent, splits, stream)


def prepare_verify_attn_mla_runs(q, kv_pool, kv_indptr, run_base, qo_indptr, kv_indptr_host, qo_indptr_host, out,
                                 lse, workspace, sm_scale, draft_mask=None, parent=None, splits=0,
                                 stream=None) -> Prepared:
    """verify_attn_mla_runs with its arguments checked and marshalled once."""
    args, keep = _run_args(q, kv_pool, kv_indptr, run_base, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
                           workspace, sm_scale, draft_mask, parent, splits, stream)
    return Prepared(_lib.verify_attn_mla_runs, "verify_attn_mla_runs", args, keep)


def _fp8_args(q, kv_pool_e4m3, kv_scale, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
              workspace, sm_scale, draft_mask=None, parent=None, splits=0, stream=None):
    kvh = _host_i32(kv_indptr_host)
    qoh = _host_i32(qo_indptr_host)
    args = (_d(q, 2, "q"), _d(kv_pool_e4m3, 1, "kv_pool_e4m3"), int(kv_pool_e4m3.shape[0]), float(kv_scale),
            _d(kv_indptr, 4, "kv_indptr"), _d(kv_indices, 4, "kv_indices"), _d(qo_indptr, 4, "qo_indptr"),
            _d(draft_mask, 8, "draft_mask"), _d(parent, 4, "parent"), kvh.ctypes.data, qoh.ctypes.data, len(kvh) - 1,
            int(q.shape[1]), float(sm_scale), int(splits), _d(out, 2, "out"), _d(lse, 4, "lse"),
            _d(workspace, 0, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    return args, (q, kv_pool_e4m3, kv_indptr, kv_indices, qo_indptr, kvh, qoh, out, lse, workspace, draft_mask, parent)


def verify_attn_mla_fp8(q, kv_pool_e4m3, kv_scale, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host,
                        out, lse, workspace, sm_scale, draft_mask=None, parent=None, splits=0, stream=None):
    """verify_attn_mla on an e4m3 latent pool ([S, 576] uint8 codes) with one scale."""
    args, _ = _fp8_args(q, kv_pool_e4m3, kv_scale, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host,
                        out, lse, workspace, sm_scale, draft_mask, parent, splits, stream)
    _check(_lib.verify_attn_mla_fp8(*args), "verify_attn_mla_fp8")


def prepare_verify_attn_mla_fp8(*a, **k) -> Prepared:
    """verify_attn_mla_fp8 with its arguments checked and marshalled once."""
    args, keep = _fp8_args(*a, **k)
    return Prepared(_lib.verify_attn_mla_fp8, "verify_attn_mla_fp8", args, keep)


def verify_attn_mla_test_fault(fault: int, wait_cycles: int = 0):
    """Failure test only: fault 1 makes the next tensor-core calls on this thread time out; 0 restores."""
    _check(_lib.verify_attn_mla_test_fault(int(fault), int(wait_cycles)), "verify_attn_mla_test_fault")


def verify_attn_mla_tree_accept(qo_indptr, parent, draft_token, target_token, root_token, accept_len, accept_path,
                                next_token, status_word=None, stream=None):
    """Greedy acceptance of the verified draft tree (device int32 arrays; parent None = chain)."""
    batch = int(qo_indptr.numel()) - 1
    rc = _lib.verify_attn_mla_tree_accept(_d(qo_indptr, 4, "qo_indptr"), _d(parent, 4, "parent"),
                                          _d(draft_token, 4, "draft_token"), _d(target_token, 4, "target_token"),
                                          _d(root_token, 4, "root_token"), batch, int(draft_token.numel()),
                                          _d(accept_len, 4, "accept_len"), _d(accept_path, 4, "accept_path"),
                                          _d(next_token, 4, "next_token"), _d(status_word, 4, "status_word"),
                                          _stream(stream))
    _check(rc, "verify_attn_mla_tree_accept")


def verify_attn_mla_simt(q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out, lse,
                         workspace, sm_scale, draft_mask=None, parent=None, splits=0, stream=None):
    """Same operation on the CUDA-core kernel."""
    _run(_lib.verify_attn_mla_simt, "verify_attn_mla_simt", q, kv_pool, kv_indptr, kv_indices, qo_indptr,
         kv_indptr_host, qo_indptr_host, out, lse, workspace, sm_scale, draft_mask, parent, splits, stream)


def verify_attn_mla_merge(o_parts, lse_parts, out, lse, stream=None):
    S, R = int(o_parts.shape[0]), int(o_parts.shape[1])
    _check(_lib.verify_attn_mla_merge(_d(o_parts, 4, "o_parts"), _d(lse_parts, 4, "lse_parts"), S, R,
                                      _d(out, 2, "out"), _d(lse, 4, "lse"), _stream(stream)), "verify_attn_mla_merge")


def verify_attn_mla_tree_mask(parent, qo_indptr, mask_out, status_word=None, stream=None):
    B = int(qo_indptr.shape[0]) - 1
    T = int(parent.shape[0])
    _check(_lib.verify_attn_mla_tree_mask(_d(parent, 4, "parent"), _d(qo_indptr, 4, "qo_indptr"), B, T,
                                          _d(mask_out, 8, "mask_out"), _d(status_word, 4, "status_word"),
                                          _stream(stream)), "verify_attn_mla_tree_mask")


def verify_attn_mla_check(workspace, stream=None) -> int:
    """Device status of the last call on `workspace` (synchronises the stream)."""
    return int(_lib.verify_attn_mla_check(_d(workspace, 0, "workspace"), _stream(stream)))


def verify_attn_mla_host_buffer_size(qo_indptr_host, kv_indptr_host, num_heads: int, splits: int = 0,
                                     has_mask: bool = False, has_parent: bool = False) -> int:
    qo = _host_i32(qo_indptr_host)
    kv = _host_i32(kv_indptr_host)
    n = ctypes.c_size_t(0)
    _check(_lib.verify_attn_mla_host_buffer_size(len(qo) - 1, num_heads, qo.ctypes.data, kv.ctypes.data, splits,
                                                 int(has_mask), int(has_parent), ctypes.byref(n)),
           "verify_attn_mla_host_buffer_size")
    return int(n.value)


def _host_args(q_host, kv_pool, kv_indptr_host, kv_indices_host, qo_indptr_host, out_host, lse_host, device_buffer,
               sm_scale, draft_mask_host=None, parent_host=None, splits=0, stream=None, num_heads=None):
    kvh = _host_i32(kv_indptr_host)
    qoh = _host_i32(qo_indptr_host)
    H = int(num_heads if num_heads is not None else q_host.shape[1])
    args = (_h(q_host, 2, "q_host"), _d(kv_pool, 2, "kv_pool"), int(kv_pool.shape[0]), kvh.ctypes.data,
            _h(kv_indices_host, 4, "kv_indices_host"), qoh.ctypes.data, _h(draft_mask_host, 8, "draft_mask_host"),
            _h(parent_host, 4, "parent_host"), len(kvh) - 1, H, float(sm_scale), int(splits),
            _h(out_host, 2, "out_host"), _h(lse_host, 4, "lse_host"), _d(device_buffer, 0, "device_buffer"),
            device_buffer.numel() * device_buffer.element_size(), _stream(stream))
    return args, (q_host, kv_pool, kvh, kv_indices_host, qoh, out_host, lse_host, device_buffer, draft_mask_host,
                  parent_host)


def verify_attn_mla_host(*a, **k):
    """Host-memory inputs/outputs, device-resident kv_pool; returns after the stream has finished."""
    args, _ = _host_args(*a, **k)
    _check(_lib.verify_attn_mla_host(*args), "verify_attn_mla_host")


def prepare_verify_attn_mla_host(*a, **k) -> Prepared:
    """verify_attn_mla_host with its arguments checked and marshalled once; call the result to run it."""
    args, keep = _host_args(*a, **k)
    return Prepared(_lib.verify_attn_mla_host, "verify_attn_mla_host", args, keep)


def verify_attn_mla_version() -> int:
    return int(_lib.verify_attn_mla_version())


def verify_attn_mla_timing_enable(capacity: int):
    _check(_lib.verify_attn_mla_timing_enable(int(capacity)), "verify_attn_mla_timing_enable")


def verify_attn_mla_timing_read(capacity: int):
    """(gather_ms, verify_ms, merge_ms) arrays of the recorded calls, in launch order."""
    g = np.zeros(max(capacity, 1), np.float32)
    v = np.zeros(max(capacity, 1), np.float32)
    m = np.zeros(max(capacity, 1), np.float32)
    n = ctypes.c_int(0)
    _check(_lib.verify_attn_mla_timing_read(g.ctypes.data, v.ctypes.data, m.ctypes.data, int(capacity),
                                            ctypes.byref(n)), "verify_attn_mla_timing_read")
    return g[: n.value].copy(), v[: n.value].copy(), m[: n.value].copy()


STATIC_SCRATCH_BYTES = 32 << 20


def verify_attn_mla_simt_static(q, kv_pool, kv_indptr, kv_indices, qo_indptr, kv_indptr_host, qo_indptr_host, out,
                                lse, sm_scale, draft_mask=None, parent=None, splits=0, stream=None):
    """CUDA-core verify with the library's fixed scratch array instead of a workspace (no allocation)."""
    kvh = _host_i32(kv_indptr_host)
    qoh = _host_i32(qo_indptr_host)
    rc = _lib.verify_attn_mla_simt_static(_d(q, 2, "q"), _d(kv_pool, 2, "kv_pool"), int(kv_pool.shape[0]),
                                          _d(kv_indptr, 4, "kv_indptr"), _d(kv_indices, 4, "kv_indices"),
                                          _d(qo_indptr, 4, "qo_indptr"), _d(draft_mask, 8, "draft_mask"),
                                          _d(parent, 4, "parent"),
                                          kvh.ctypes.data, qoh.ctypes.data, len(kvh) - 1, int(q.shape[1]),
                                          float(sm_scale), int(splits), _d(out, 2, "out"), _d(lse, 4, "lse"),
                                          _stream(stream))
    _check(rc, "verify_attn_mla_simt_static")


def verify_attn_mla_simt_static_check(stream=None) -> int:
    """Synchronises the stream and returns the status word the static-scratch calls left (0 = ok)."""
    return int(_lib.verify_attn_mla_simt_static_check(_stream(stream)))
