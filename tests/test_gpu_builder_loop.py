"""The whole hot path over many iterations: the library's stall-free builder
forms each hybrid batch, the KV append writes its new tokens into a
persistent page pool, and attention runs over it; every iteration is checked
against the oracle (oracle append on its own copy of the pool, oracle
attention) — append bit-exact, attention within max-abs 1e-2 / mean-abs 1e-3."""
import math

import numpy as np
import pytest
import torch

from _gpu import compare
from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from chunked_prefill_decode_gb300.device import device_batch
from oracle import paged_attention as pa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("geom,budget,n_req,seed", [
    ((32, 8, 128), 64, 10, 0),
    ((8, 8, 64), 24, 8, 1),
    ((56, 8, 128), 128, 6, 2),
])
def test_builder_driven_iterations(geom, budget, n_req, seed):
    hb = lib()
    hq, hkv, d = geom
    P, num_pages, maxp = 16, 400, 40
    rng = np.random.default_rng(seed)
    order = rng.permutation(num_pages)
    b = hb.Builder(budget, P, num_pages, maxp, page_order=order)
    arrivals = sorted(rng.integers(0, 12, size=n_req).tolist())
    reqs = [(i, int(rng.integers(1, 300)), int(rng.integers(1, 12))) for i in range(n_req)]
    stream = list(zip(arrivals, reqs))
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(seed)
    # pool starts as NaN sentinels everywhere (nothing cached yet)
    sentinel = torch.full((num_pages, P, hkv, d), workloads.SENTINEL_BITS, dtype=torch.int16)
    k_pool = sentinel.view(torch.bfloat16).clone().to(dev)
    v_pool = sentinel.view(torch.bfloat16).clone().to(dev)
    k_ref = workloads.bf16_bits(k_pool)
    v_ref = workloads.bf16_bits(v_pool)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    scale = 1.0 / math.sqrt(d)
    it, checked = 0, 0
    while it < 200:
        while stream and stream[0][0] <= it:
            _, (rid, p, m) = stream.pop(0)
            b.add_request(rid, p, m)
        it += 1
        batch = b.step()
        if batch is None:
            if not stream and b.counts()[:2] == (0, 0):
                break
            continue
        ql, cl, bt = batch["q_len"], batch["context_len"], batch["block_table"]
        T = int(ql.sum())
        q = torch.randn(T, hq, d, generator=g).to(torch.bfloat16)
        kn = torch.randn(T, hkv, d, generator=g).to(torch.bfloat16)
        vn = torch.randn(T, hkv, d, generator=g).to(torch.bfloat16)
        db = device_batch(ql, cl, bt, num_pages, hq, hkv, d, P, dev)
        out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev)
        hb.hb_kv_append(db.batch, kn.to(dev), vn.to(dev), k_pool, v_pool)
        plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms)
        hb.hb_attention(db.batch, plan, q.to(dev), k_pool, v_pool, scale, out, ws)
        hb.hb_check()
        # oracle on its own pool copy
        bits = workloads.bf16_bits
        k_ref, v_ref = pa.kv_append(k_ref, v_ref, bits(kn), bits(vn), ql, cl, bt, P)
        assert np.array_equal(bits(k_pool), k_ref) and np.array_equal(bits(v_pool), v_ref)
        ref = pa.attention(bits(q), k_ref, v_ref, ql, cl, bt, P, hq, hkv, scale)
        compare(out, ref)
        b.complete()
        checked += 1
    assert checked >= 5 and not stream
