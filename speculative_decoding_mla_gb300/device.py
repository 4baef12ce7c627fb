"""Device-side plumbing for the binding: moves a synth.Case into HBM with torch,
allocates outputs and the workspace, and calls the C ABI.  torch provides
memory and streams only; no step of the operation runs here."""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import binding


@dataclass
class DeviceCase:
    q: torch.Tensor            # [T, H, 576] bf16
    kv_pool: torch.Tensor      # [S, 576] bf16
    kv_indptr: torch.Tensor    # [B+1] int32
    kv_indices: torch.Tensor   # [N] int32
    qo_indptr: torch.Tensor    # [B+1] int32
    parent: Optional[torch.Tensor]
    draft_mask: Optional[torch.Tensor]
    kv_indptr_host: np.ndarray
    qo_indptr_host: np.ndarray
    sm_scale: float

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])


def _u16_to_bf16(a: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_device(case, device="cuda", draft_mask: Optional[np.ndarray] = None, use_parent: bool = True) -> DeviceCase:
    dev = torch.device(device)
    par = None
    if use_parent and case.parent is not None and draft_mask is None:
        par = torch.from_numpy(np.ascontiguousarray(case.parent, np.int32)).to(dev)
    dm = None
    if draft_mask is not None:
        dm = torch.from_numpy(np.ascontiguousarray(draft_mask, np.uint64).view(np.int64)).to(dev)
    return DeviceCase(
        q=_u16_to_bf16(case.q, dev),
        kv_pool=_u16_to_bf16(case.kv_pool, dev),
        kv_indptr=torch.from_numpy(np.ascontiguousarray(case.kv_indptr, np.int32)).to(dev),
        kv_indices=torch.from_numpy(np.ascontiguousarray(case.kv_indices, np.int32)).to(dev),
        qo_indptr=torch.from_numpy(np.ascontiguousarray(case.qo_indptr, np.int32)).to(dev),
        parent=par, draft_mask=dm,
        kv_indptr_host=np.ascontiguousarray(case.kv_indptr, np.int32),
        qo_indptr_host=np.ascontiguousarray(case.qo_indptr, np.int32),
        sm_scale=float(case.sm_scale))


def alloc_outputs(dc: DeviceCase):
    T, H = dc.total_q, dc.num_heads
    out = torch.empty((T, H, binding.D_V), dtype=torch.bfloat16, device=dc.q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=dc.q.device)
    return out, lse


def alloc_workspace(dc: DeviceCase, splits: int = 0) -> torch.Tensor:
    n = binding.verify_attn_mla_workspace_size(dc.qo_indptr_host, dc.kv_indptr_host, dc.num_heads, splits)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=dc.q.device)


def run(dc: DeviceCase, kernel: str = "tc", splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """One verify call; returns (out, lse, workspace)."""
    if out is None or lse is None:
        out, lse = alloc_outputs(dc)
    if workspace is None:
        workspace = alloc_workspace(dc, splits)
    fn = binding.verify_attn_mla if kernel == "tc" else binding.verify_attn_mla_simt
    fn(dc.q, dc.kv_pool, dc.kv_indptr, dc.kv_indices, dc.qo_indptr, dc.kv_indptr_host, dc.qo_indptr_host, out, lse,
       workspace, dc.sm_scale, draft_mask=dc.draft_mask, parent=dc.parent, splits=splits, stream=stream)
    return out, lse, workspace


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)
