"""The no-allocation decode entry point against the workspace path (GPU).

hb_decode_attention_noalloc is for callers that cannot allocate device
memory (an engine that has handed its free HBM to the KV-cache pool, a
plugin given raw pointers only): it keeps its scratch in a fixed array inside
the library.  Its output must match hb_plan + hb_attention on the same
decode-row batch, on two calls in a row (the second call finds the first
call's leftovers in the shared array).  This file is collected last, so a
run that stops at the first failure has already run every other test.
"""
import math

import numpy as np
import pytest
import torch

from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from chunked_prefill_decode_gb300.device import device_batch
from chunked_prefill_decode_gb300.workloads import Shape, layout_from_rows

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def _setup(rows, geom, seed):
    hb = lib()
    lay = layout_from_rows(Shape(*geom), rows, seed)
    ten = workloads.make_tensors(lay, seed)
    sh = lay.shape
    dev = torch.device("cuda:0")
    db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                      sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev)
    q = ten.q.to(dev)
    kc, vc = ten.k_cache.to(dev), ten.v_cache.to(dev)
    hb.hb_kv_append(db.batch, ten.k_new.to(dev), ten.v_new.to(dev), kc, vc)
    return hb, lay, db, q, kc, vc, 1.0 / math.sqrt(sh.head_dim)


@pytest.mark.parametrize("rows,geom", [
    ([(1, int(c)) for c in np.random.default_rng(7).integers(1, 6000, size=48)], (32, 8, 128)),
    ([(1, 9000), (1, 3), (1, 700), (1, 16)], (56, 8, 128)),
    ([(1, int(c)) for c in np.random.default_rng(8).integers(1, 900, size=20)], (8, 8, 64)),
])
def test_noalloc_matches_workspace_path_twice(rows, geom):
    hb, lay, db, q, kc, vc, scale = _setup(rows, geom, 21)
    ref = torch.empty_like(q)
    plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len,
                          torch.cuda.get_device_properties(0).multi_processor_count)
    hb.hb_attention(db.batch, plan, q, kc, vc, scale, ref, ws)
    hb.hb_check()
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        hb.hb_decode_attention_noalloc(db.batch, db.q_len, db.context_len, q, kc, vc,
                                       scale, out)
        hb.hb_check()
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_noalloc_rejects_chunk_rows_and_too_many_items():
    hb, lay, db, q, kc, vc, scale = _setup([(1, 50), (7, 90)], (32, 8, 128), 22)
    out = torch.empty_like(q)
    with pytest.raises(hb.HbError) as e:
        hb.hb_decode_attention_noalloc(db.batch, db.q_len, db.context_len, q, kc, vc,
                                       scale, out)
    assert e.value.status == 3
    # 4100 decode rows with one kv block each need more than 4096 items
    hb, lay, db, q, kc, vc, scale = _setup([(1, 2)] * 4100, (8, 8, 64), 23)
    out = torch.empty_like(q)
    with pytest.raises(hb.HbError) as e:
        hb.hb_decode_attention_noalloc(db.batch, db.q_len, db.context_len, q, kc, vc,
                                       scale, out)
    assert e.value.status == 4
