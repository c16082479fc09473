"""Move a batch's int32 descriptors to the GPU and wrap them for the C ABI.

Plumbing only (torch owns the device memory): the arrays are copied as they
are, cu_q_len is the prefix sum of q_len, and the returned object keeps the
tensors alive as long as its hb_batch is in use.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import hb


@dataclass
class DeviceBatch:
    batch: hb.HbBatch
    q_len: np.ndarray            # host copies, as hb_plan wants them
    context_len: np.ndarray
    cu_q_len: torch.Tensor       # device
    context_len_d: torch.Tensor
    block_table: torch.Tensor


def device_batch(q_len, context_len, block_table, num_pages, num_q_heads,
                 num_kv_heads, head_dim, page_size=16, device="cuda",
                 non_blocking=False, sliding_window=0) -> DeviceBatch:
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    cl = np.ascontiguousarray(context_len, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    if bt.ndim != 2 or bt.shape[0] != ql.shape[0]:
        raise ValueError("block_table must be [num_seqs, max_pages_per_seq]")
    cu = np.zeros(ql.shape[0] + 1, dtype=np.int32)
    np.cumsum(ql, out=cu[1:])
    cu_d = torch.from_numpy(cu).to(device, non_blocking=non_blocking)
    cl_d = torch.from_numpy(cl).to(device, non_blocking=non_blocking)
    bt_d = torch.from_numpy(bt).to(device, non_blocking=non_blocking)
    b = hb.make_batch(ql.shape[0], int(cu[-1]), max(1, bt.shape[1]), num_pages,
                      num_q_heads, num_kv_heads, head_dim, cu_d, cl_d, bt_d,
                      page_size=page_size, sliding_window=sliding_window)
    return DeviceBatch(b, ql, cl, cu_d, cl_d, bt_d)


def from_layout(layout, device="cuda") -> DeviceBatch:
    """DeviceBatch of a workloads.BatchLayout."""
    sh = layout.shape
    return device_batch(layout.q_len, layout.context_len, layout.block_table,
                        layout.num_pages, sh.num_q_heads, sh.num_kv_heads,
                        sh.head_dim, sh.page_size, device,
                        sliding_window=sh.sliding_window)
