"""Pins of the stall-free batch-builder oracle (CPU only): a hand-worked
trace and the invariants the pages state, over random request streams."""
import json
import os

import numpy as np
import pytest

from oracle.stall_free import OutOfPages, StallFreeBuilder

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run_trace(b, n_max=1000):
    out = []
    for _ in range(n_max):
        batch = b.step()
        if batch is None:
            out.append(None)
            return out
        rows = [[r.rid, r.kind, r.q_len, r.context_len, r.pages] for r in batch.rows]
        fin = b.complete(batch)
        out.append({"rows": rows, "over_budget": batch.over_budget,
                    "finished": fin, "free_after": list(b.free)})
    raise AssertionError("builder did not drain")


def test_hand_worked_trace():
    with open(os.path.join(GOLDEN, "stall_free_trace_a.json")) as f:
        g = json.load(f)
    b = StallFreeBuilder(g["budget"], g["page_size"], g["num_pages"],
                         g["max_pages_per_seq"])
    for rid, prompt, max_new in g["requests"]:
        b.add_request(rid, prompt, max_new)
    assert _run_trace(b) == g["iterations"]


def _random_stream(seed, budget, page, num_pages, n_req, max_prompt, max_new):
    rng = np.random.default_rng(seed)
    b = StallFreeBuilder(budget, page, num_pages, 64)
    arrivals = sorted(rng.integers(0, 40, size=n_req).tolist())
    reqs = [(i, int(rng.integers(1, max_prompt + 1)), int(rng.integers(1, max_new + 1)))
            for i in range(n_req)]
    return rng, b, list(zip(arrivals, reqs))


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("budget", [1, 7, 16, 64])
def test_invariants_on_random_streams(seed, budget):
    page, num_pages = 4, 200
    rng, b, stream = _random_stream(seed, budget, page, num_pages, 25, 90, 12)
    done_prefill = {}
    admitted_order = []
    it = 0
    prompt = {rid: p for _, (rid, p, _) in stream}
    max_new = {rid: m for _, (rid, _, m) in stream}
    gen = {}
    while True:
        while stream and stream[0][0] <= it:
            _, (rid, p, m) = stream.pop(0)
            b.add_request(rid, p, m)
        decoding = {r.rid for r in b.running if r.phase == "decode"}
        batch = b.step()
        it += 1
        if batch is None:
            if not stream and not b.waiting and not b.running:
                break
            continue
        rows = batch.rows
        kinds = [r.kind for r in rows]
        # decodes are all present, first, one token each
        assert {r.rid for r in rows if r.kind == "decode"} == decoding
        assert kinds == sorted(kinds, key=lambda k: k != "decode")
        assert all(r.q_len == 1 for r in rows if r.kind == "decode")
        # budget
        if batch.over_budget:
            assert all(k == "decode" for k in kinds)
        else:
            assert batch.num_tokens <= budget
        # pages: disjoint ownership and enough to hold the context
        owned = [p for r in rows for p in r.pages]
        assert len(owned) == len(set(owned))
        assert not set(owned) & set(b.free)
        for r in rows:
            assert len(r.pages) == -(-r.context_len // page)
        # chunks continue where the prompt left off
        for r in rows:
            if r.kind == "prefill":
                before = done_prefill.get(r.rid, 0)
                assert r.context_len == before + r.q_len
                if before == 0:
                    admitted_order.append(r.rid)
                done_prefill[r.rid] = before + r.q_len
                assert done_prefill[r.rid] <= prompt[r.rid]
            else:
                gen[r.rid] = gen.get(r.rid, 1) + 1
                assert r.context_len == prompt[r.rid] + gen[r.rid] - 1
        b.complete(batch)
        assert it < 5000
    # every prompt was prefilled exactly once, in arrival (FCFS) order
    assert all(done_prefill[rid] == prompt[rid] for rid in prompt)
    assert admitted_order == sorted(prompt)
    assert all(gen.get(rid, 1) == max_new[rid] for rid in prompt)
    assert sorted(b.free) == list(range(num_pages))


def test_decodes_over_budget_still_scheduled():
    b = StallFreeBuilder(2, 4, 64, 16)
    for i in range(4):
        b.add_request(i, 1, 5)
    bt = b.step()            # admits 2 one-token prompts
    b.complete(bt)
    bt = b.step()            # 2 decodes fill the budget; nothing admitted
    assert [r.kind for r in bt.rows] == ["decode", "decode"]
    b.complete(bt)
    b.budget = 1             # decodes alone now exceed the budget
    bt = b.step()
    assert [r.kind for r in bt.rows] == ["decode", "decode"] and bt.over_budget


def test_admission_stops_at_first_request_without_pages():
    b = StallFreeBuilder(100, 4, 5, 16)
    b.add_request(0, 12, 1)   # 3 pages
    b.add_request(1, 12, 1)   # needs 3 pages, only 2 left -> stop
    b.add_request(2, 4, 1)    # would fit, but FCFS does not skip
    bt = b.step()
    assert [r.rid for r in bt.rows] == [0]


def test_decode_without_free_page_is_an_error():
    b = StallFreeBuilder(100, 4, 1, 16)
    b.add_request(0, 4, 3)
    b.complete(b.step())
    with pytest.raises(OutOfPages):
        b.step()
