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


def _raw_step(hb, b, max_rows):
    import ctypes
    mp = b.max_pages_per_seq
    out = {"q_len": np.zeros(max(max_rows, 1), np.int32),
           "context_len": np.zeros(max(max_rows, 1), np.int32),
           "block_table": np.zeros((max(max_rows, 1), mp), np.int32),
           "ids": np.zeros(max(max_rows, 1), np.int64),
           "kind": np.zeros(max(max_rows, 1), np.int32)}
    n, over = ctypes.c_int32(0), ctypes.c_int32(0)
    st = hb.load().hb_builder_step(b._h, max_rows, ctypes.byref(n), hb._ptr(out["q_len"]),
                                   hb._ptr(out["context_len"]), hb._ptr(out["block_table"]),
                                   hb._ptr(out["ids"]), hb._ptr(out["kind"]), ctypes.byref(over))
    return st, n.value


def test_failed_step_leaves_the_builder_unchanged():
    """A step refused for too few output rows puts back every page it took:
    the free list, the counts and the next batch are those of a twin builder
    that never failed."""
    hb = lib()
    order = np.random.default_rng(5).permutation(200)
    a = hb.Builder(64, 16, 200, 16, page_order=order)
    twin = hb.Builder(64, 16, 200, 16, page_order=order)
    for b in (a, twin):
        for rid in range(6):
            b.add_request(rid, 10 + 7 * rid, 3)
    for _ in range(2):                       # some decodes running, prefills ongoing
        assert a.step() is not None and twin.step() is not None
        assert a.complete() == twin.complete()
    before = (a.free_list(), a.counts())
    st, need = _raw_step(hb, a, 1)
    assert st == 4 and need > 1              # HB_ERR_WORKSPACE, rows needed reported
    assert (a.free_list(), a.counts()) == before
    x, y = a.step(), twin.step()
    for k in ("q_len", "context_len", "block_table", "ids", "kind"):
        assert x[k].tolist() == y[k].tolist()
    assert a.complete() == twin.complete()
    assert a.free_list() == twin.free_list()


def test_decode_out_of_pages_leaves_the_builder_unchanged():
    hb = lib()
    b = hb.Builder(8, 4, 3, 8)
    b.add_request(1, 4, 10)                  # one 4-token page per prompt
    b.add_request(2, 4, 10)
    b.step()
    b.complete()                             # both prefilled, one page free
    before = (b.free_list(), b.counts())
    assert before == ([2], (0, 2, 1))
    for _ in range(2):
        # both decode at context 5: request 1 takes the free page, then
        # request 2 finds none; the step takes nothing in the end
        with pytest.raises(hb.HbError) as e:
            b.step()
        assert e.value.status == 8
        assert (b.free_list(), b.counts()) == before


def test_step_cost_does_not_grow_with_the_pool():
    """Forming a batch costs what its rows cost: 64 decodes and a chunk
    take about as long with two million free pages as with two thousand."""
    import statistics
    import time
    hb = lib()

    def median_step_us(num_pages):
        b = hb.Builder(512, 16, num_pages, 64)
        for rid in range(64):
            b.add_request(rid, 16, 200)
        b.add_request(999, 900, 1)
        ts = []
        for _ in range(40):
            t = time.perf_counter()
            b.step()
            b.complete()
            ts.append(time.perf_counter() - t)
        return statistics.median(ts[5:]) * 1e6

    small, big = median_step_us(2000), median_step_us(2_000_000)
    assert big < 20 * small + 200, (small, big)
