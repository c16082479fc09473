"""The library's C++ stall-free builder against the oracle builder (CPU)."""
import json
import os

import numpy as np
import pytest

from _hbutil import lib
from oracle.stall_free import OutOfPages, StallFreeBuilder

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _native_trace(b, max_pages):
    out = []
    for _ in range(1000):
        bt = b.step()
        if bt is None:
            out.append(None)
            return out
        rows = []
        for i in range(len(bt["q_len"])):
            pages = [int(p) for p in bt["block_table"][i] if p >= 0]
            rows.append([int(bt["ids"][i]), "decode" if bt["kind"][i] == 0 else "prefill",
                         int(bt["q_len"][i]), int(bt["context_len"][i]), pages])
        fin = b.complete()
        out.append({"rows": rows, "over_budget": bt["over_budget"], "finished": fin,
                    "free_after": b.free_list()})
    raise AssertionError("builder did not drain")


def test_native_builder_hand_worked_trace():
    hb = lib()
    with open(os.path.join(GOLDEN, "stall_free_trace_a.json")) as f:
        g = json.load(f)
    b = hb.Builder(g["budget"], g["page_size"], g["num_pages"], g["max_pages_per_seq"])
    for rid, prompt, max_new in g["requests"]:
        b.add_request(rid, prompt, max_new)
    assert _native_trace(b, g["max_pages_per_seq"]) == g["iterations"]


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("budget,num_pages", [(1, 300), (13, 300), (64, 60), (512, 2000)])
def test_native_matches_oracle_on_random_streams(seed, budget, num_pages):
    hb = lib()
    rng = np.random.default_rng(seed)
    page, maxp = 16, 64
    order = rng.permutation(num_pages)
    nb = hb.Builder(budget, page, num_pages, maxp, page_order=order)
    ob = StallFreeBuilder(budget, page, num_pages, maxp, page_order=order)
    arrivals = sorted(rng.integers(0, 30, size=30).tolist())
    max_prompt = 600 if budget >= 64 else 60
    reqs = [(i, int(rng.integers(1, max_prompt)), int(rng.integers(1, 40))) for i in range(30)]
    stream = list(zip(arrivals, reqs))
    it = 0
    while True:
        while stream and stream[0][0] <= it:
            _, (rid, p, m) = stream.pop(0)
            nb.add_request(rid, p, m)
            ob.add_request(rid, p, m)
        it += 1
        try:
            ob_batch = ob.step()
            o_err = None
        except OutOfPages as e:
            o_err = e
        if o_err is not None:
            with pytest.raises(hb.HbError) as ei:
                nb.step()
            assert ei.value.status == 8
            return
        n_batch = nb.step()
        if ob_batch is None:
            assert n_batch is None
            if not stream and not ob.waiting and not ob.running:
                break
            continue
        assert n_batch is not None
        assert n_batch["over_budget"] == ob_batch.over_budget
        assert n_batch["ids"].tolist() == [r.rid for r in ob_batch.rows]
        assert n_batch["q_len"].tolist() == [r.q_len for r in ob_batch.rows]
        assert n_batch["context_len"].tolist() == [r.context_len for r in ob_batch.rows]
        assert n_batch["kind"].tolist() == [0 if r.kind == "decode" else 1 for r in ob_batch.rows]
        assert n_batch["block_table"].tolist() == ob_batch.block_table(maxp)
        assert nb.complete() == ob.complete(ob_batch)
        assert nb.free_list() == list(ob.free)
        assert it < 20000


def test_native_builder_argument_errors():
    hb = lib()
    with pytest.raises(hb.HbError):
        hb.Builder(0, 16, 10, 4)
    b = hb.Builder(8, 16, 10, 4)
    with pytest.raises(hb.HbError) as e:
        b.add_request(1, 0, 1)
    assert e.value.status == 2
    with pytest.raises(hb.HbError) as e:
        b.add_request(1, 60, 10)        # 69 tokens > 4 pages of 16
    assert e.value.status == 2
    b.add_request(1, 5, 2)
    with pytest.raises(hb.HbError) as e:
        b.add_request(1, 5, 2)
    assert e.value.status == 1
    assert b.counts() == (1, 0, 10)
