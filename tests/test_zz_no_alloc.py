"""The no-allocation decode entry point, checked against the CPU oracle and
the workspace path (GPU).

hb_decode_attention_noalloc is for callers that cannot allocate device
memory (an engine that has handed its free HBM to the KV-cache pool, a
plugin given raw pointers only): it keeps its scratch in a fixed array inside
the library.  Its output must equal the fp64 oracle within the attention
bounds and agree with hb_plan + hb_attention on the same decode-row batch,
also on a call that follows a larger call of another shape (which leaves its
items, counters and partial states in the shared array).  Repeated calls
must leave the device's free memory unchanged.  This file is collected last,
so a run that stops at the first failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from _gpu import compare, oracle_step, sms
from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from chunked_prefill_decode_gb300.device import device_batch
from chunked_prefill_decode_gb300.workloads import Shape, layout_from_rows

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3
SCRATCH_BYTES = 8 * 1024 * 1024     # HB_NOALLOC_SCRATCH_BYTES


class Case:
    """One decode-row batch on cuda:0 with its caches after the append, its
    output buffer and the oracle's answer."""

    def __init__(self, rows, geom, seed, window=0):
        hb = lib()
        self.hb = hb
        lay = layout_from_rows(Shape(*geom, sliding_window=window), rows, seed)
        ten = workloads.make_tensors(lay, seed)
        sh = lay.shape
        dev = torch.device("cuda:0")
        self.lay = lay
        self.db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                               sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev,
                               sliding_window=window)
        self.q = ten.q.to(dev)
        self.kc, self.vc = ten.k_cache.to(dev), ten.v_cache.to(dev)
        hb.hb_kv_append(self.db.batch, ten.k_new.to(dev), ten.v_new.to(dev), self.kc, self.vc)
        self.scale = 1.0 / math.sqrt(sh.head_dim)
        self.out = torch.empty_like(self.q)
        _, _, self.ref = oracle_step(lay, ten)
        hb.hb_check()

    def noalloc(self):
        self.out.fill_(float("nan"))
        self.hb.hb_decode_attention_noalloc(self.db.batch, self.db.q_len, self.db.context_len,
                                            self.q, self.kc, self.vc, self.scale, self.out)
        self.hb.hb_check()
        return self.out

    def workspace_path(self):
        out = torch.empty_like(self.q)
        plan, ws = self.hb.hb_plan(self.db.batch, self.db.q_len, self.db.context_len, sms())
        self.hb.hb_attention(self.db.batch, plan, self.q, self.kc, self.vc, self.scale, out, ws)
        self.hb.hb_check()
        return out

    def full_grid_plan(self):
        """Header of the workspace path's host plan (one decode CTA per SM)."""
        plan, _ = self.hb.hb_plan(self.db.batch, self.db.q_len, self.db.context_len, sms(),
                                  upload=False)
        return self.hb.plan_header(plan)


def _rows(seed, n, lo, hi):
    return [(1, int(c)) for c in np.random.default_rng(seed).integers(lo, hi, size=n)]


CASES = [
    (_rows(7, 48, 1, 6000), (32, 8, 128), 0),
    ([(1, 9000), (1, 3), (1, 700), (1, 16)], (56, 8, 128), 0),
    (_rows(8, 20, 1, 900), (8, 8, 64), 0),
    (_rows(9, 24, 1, 5000), (32, 8, 128), 300),
    ([(1, 1), (1, 17), (1, 700), (1, 3000)], (56, 8, 128), 7),
]


@pytest.mark.parametrize("rows,geom,window", CASES)
def test_noalloc_matches_oracle_and_workspace_path(rows, geom, window):
    a = Case(rows, geom, 21, window)
    ref_ws = a.workspace_path()
    compare(ref_ws, a.ref)
    for _ in range(2):
        out = a.noalloc()
        compare(out, a.ref)
        err = (out.float() - ref_ws.float()).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_noalloc_after_a_larger_call_of_another_shape():
    """A call on batch A, then on a larger batch B of another head geometry
    with many rows split over several CTAs (its items, counters and partial
    states fill more of the shared array), then on A again: both A calls
    match the oracle."""
    a = Case(_rows(31, 12, 1, 3000), (32, 8, 128), 31)
    b = Case(_rows(32, 64, 2000, 9000), (56, 8, 128), 32)
    assert b.full_grid_plan()["num_merge_counters"] > 0
    compare(a.noalloc(), a.ref)
    compare(b.noalloc(), b.ref)
    compare(a.noalloc(), a.ref)


def test_noalloc_spreads_work_when_partial_states_overflow():
    """128 q / 32 kv heads (66.5 KB of partial state per split piece) over
    long rows: at one CTA per SM the pieces' states exceed the static array,
    so the call runs the rows over fewer, longer ranges -- and still matches
    the oracle and the workspace path."""
    c = Case(_rows(33, 24, 3500, 4500), (128, 32, 128), 33)
    hdr = c.full_grid_plan()
    slot_bytes = 128 * 128 * 4 + 128 * 8
    assert hdr["num_partial_slots"] * slot_bytes > SCRATCH_BYTES
    out = c.noalloc()
    compare(out, c.ref)
    err = (out.float() - c.workspace_path().float()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_noalloc_allocates_no_device_memory():
    """After the first call (which may load the kernel), repeated calls leave
    the device's free memory where it was."""
    c = Case(_rows(34, 40, 1, 6000), (32, 8, 128), 34)
    c.noalloc()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        c.noalloc()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    compare(c.out, c.ref)


def test_noalloc_refuses_capture_chunk_rows_and_too_many_items():
    hb = lib()
    c = Case([(1, 50), (1, 90)], (32, 8, 128), 22)
    # a call inside a stream capture is refused (its work list is copied from
    # host memory at the call); the stream stays usable afterwards
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(hb.HbError) as e:
        with torch.cuda.graph(g, stream=s):
            hb.hb_decode_attention_noalloc(c.db.batch, c.db.q_len, c.db.context_len, c.q,
                                           c.kc, c.vc, c.scale, c.out, stream=s)
    assert e.value.status == 3
    compare(c.noalloc(), c.ref)

    lay = layout_from_rows(Shape(32, 8, 128), [(1, 50), (7, 90)], 22)
    ten = workloads.make_tensors(lay, 22)
    dev = torch.device("cuda:0")
    db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                      32, 8, 128, 16, dev)
    q, kc, vc = ten.q.to(dev), ten.k_cache.to(dev), ten.v_cache.to(dev)
    with pytest.raises(hb.HbError) as e:
        hb.hb_decode_attention_noalloc(db.batch, db.q_len, db.context_len, q, kc, vc,
                                       0.1, torch.empty_like(q))
    assert e.value.status == 3
    # 4100 decode rows with one kv block each need more than 4096 items
    lay = layout_from_rows(Shape(8, 8, 64), [(1, 2)] * 4100, 23)
    ten = workloads.make_tensors(lay, 23)
    db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                      8, 8, 64, 16, dev)
    q, kc, vc = ten.q.to(dev), ten.k_cache.to(dev), ten.v_cache.to(dev)
    with pytest.raises(hb.HbError) as e:
        hb.hb_decode_attention_noalloc(db.batch, db.q_len, db.context_len, q, kc, vc,
                                       0.125, torch.empty_like(q))
    assert e.value.status == 4
