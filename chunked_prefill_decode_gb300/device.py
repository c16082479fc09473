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


class StepStaging:
    """One step's inputs (q, k_new, v_new and the batch descriptors) and its
    output, each laid out back to back in one pinned host buffer and one
    device buffer, so that a step crosses the host link with one copy each
    way.  Fill the host views (h_q, h_k_new, h_v_new, h_cu_q_len,
    h_context_len, h_block_table), call upload(stream), run the step on the
    device views (q, k_new, v_new, out and the hb_batch `batch`), then
    download(stream) into h_out.  Two instances let one step's copies
    overlap the neighbouring steps' kernels."""

    _ALIGN = 256

    @staticmethod
    def layout(num_seqs, total_q, max_pages_per_seq, num_q_heads, num_kv_heads, head_dim):
        """[(name, shape, dtype, offset, bytes)] of the packed input block (the
        same as hb_step_layout's: 256-byte aligned sections), and its size."""
        a = StepStaging._ALIGN
        parts = [("q", (total_q, num_q_heads, head_dim), torch.bfloat16),
                 ("k_new", (total_q, num_kv_heads, head_dim), torch.bfloat16),
                 ("v_new", (total_q, num_kv_heads, head_dim), torch.bfloat16),
                 ("cu_q_len", (num_seqs + 1,), torch.int32),
                 ("context_len", (num_seqs,), torch.int32),
                 ("block_table", (num_seqs, max_pages_per_seq), torch.int32)]
        offs, off = [], 0
        for name, shape, dt in parts:
            n = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
            offs.append((name, shape, dt, off, n))
            off = (off + n + a - 1) // a * a
        return offs, off

    def __init__(self, num_seqs, total_q, max_pages_per_seq, num_pages, num_q_heads,
                 num_kv_heads, head_dim, page_size=16, sliding_window=0, device="cuda"):
        offs, off = self.layout(num_seqs, total_q, max_pages_per_seq, num_q_heads,
                                num_kv_heads, head_dim)
        self.in_bytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=device)

        def view(buf, o, n, shape, dt):
            return buf[o:o + n].view(dt).view(shape)
        for name, shape, dt, o, n in offs:
            setattr(self, "h_" + name, view(self.host, o, n, shape, dt))
            setattr(self, name, view(self.dev, o, n, shape, dt))
        self.out = torch.empty(total_q, num_q_heads, head_dim, dtype=torch.bfloat16, device=device)
        self.h_out = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        self.out_bytes = self.out.numel() * 2
        self.batch = hb.make_batch(num_seqs, total_q, max(1, max_pages_per_seq), num_pages,
                                   num_q_heads, num_kv_heads, head_dim, self.cu_q_len,
                                   self.context_len, self.block_table, page_size=page_size,
                                   sliding_window=sliding_window)

    def step_buffers(self, plan, workspace):
        """hb_step's buffers over this staging (plan: host uint8 array,
        workspace: device uint8 tensor, both sized by hb_plan)."""
        b = hb.HbStepBuffers()
        b.h_in, b.d_in = self.host.data_ptr(), self.dev.data_ptr()
        b.h_out, b.d_out = self.h_out.data_ptr(), self.out.data_ptr()
        b.h_plan, b.plan_bytes = plan.ctypes.data, plan.nbytes
        b.d_workspace, b.workspace_bytes = workspace.data_ptr(), workspace.numel()
        return b

    def upload(self, stream=None):
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            self.dev.copy_(self.host, non_blocking=True)

    def download(self, stream=None):
        with torch.cuda.stream(stream or torch.cuda.current_stream()):
            self.h_out.copy_(self.out, non_blocking=True)
