"""Moving synthetic cases onto the GPU and running them through the C ABI.

Used by the GPU tests only.  Inputs come from ``workloads``; the expected
values come from ``oracle``; the computation under test is the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch

import paged_split_kv_attn_gb300 as pskv
import workloads as W

TOL = 2e-3  # max |out - fp64 reference| for fp32 accumulation (pegainfer #1055 gate)


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    """numpy data (bf16 bits as uint16, or float32) -> CUDA tensor of that type."""
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.astype(np.float32, copy=False)).cuda()


def i32(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, np.int32)).cuda()


class DevCase:
    """A PagedCase with its arrays on the device and a layout over its pools."""

    def __init__(self, case: W.PagedCase):
        self.case = case
        self.k_pool = to_dev(case.k_pool, case.dtype)
        self.v_pool = to_dev(case.v_pool, case.dtype)
        self.q = to_dev(case.q, case.dtype)
        self.tables = i32(case.page_tables)
        self.lens = i32(case.seq_lens)
        self.status = torch.zeros(4, dtype=torch.int32, device="cuda")
        self.layout = pskv.paged_kv_layout_create(self.k_pool, self.v_pool, self.status)  # folded if K is narrower
        self.first_pos = None if case.first_pos is None else i32(case.first_pos)
        self.window_lo = None if case.window_lo is None else i32(case.window_lo)

    def decode(self, num_splits=0, out_dtype=torch.float32, windowed=None, **kw):
        c = self.case
        windowed = (c.window_lo is not None) if windowed is None else windowed
        if windowed:
            return pskv.decode_attn_windowed(self.layout, self.q, self.tables, self.lens,
                                             c.seq_lens, self.first_pos, self.window_lo, c.scale,
                                             num_splits=num_splits, out_dtype=out_dtype, **kw)
        return pskv.decode_attn_splitkv(self.layout, self.q, self.tables, self.lens, c.seq_lens,
                                        c.scale, num_splits=num_splits, out_dtype=out_dtype, **kw)

    def faults(self) -> int:
        torch.cuda.synchronize()
        return int(self.status[0].item())


def max_err(out: torch.Tensor, ref: np.ndarray) -> float:
    return float(np.abs(out.float().cpu().numpy().astype(np.float64) - ref).max())


def bf16_of(out_f32: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even bf16 of an fp32 output (what the bf16 output must equal)."""
    return out_f32.to(torch.bfloat16)
