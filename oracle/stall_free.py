"""Oracle for the stall-free batch builder (the iteration scheduler).

TEST INFRASTRUCTURE: a step-by-step Python statement of the scheduler that
forms each hybrid batch; only `tests/` use it.  The C++ builder in the
library is checked against it trace by trace.

Steps, in the order the pages give them ("Sarathi-Serve：以 chunked-prefills
与 stall-free batching 驯服 LLM 推理的吞吐—延迟权衡", §核心机制 2; "Sarathi-Serve:
Chunked Prefills for Stall-Free LLM Inference", "The mechanism" and
"Algorithm / figure walkthrough" steps 2-4):
  1. put one decode token of every running request that has finished its
     prefill into the batch;
  2. continue the unfinished prefills with a chunk each, as far as the token
     budget B allows;
  3. admit waiting requests, cutting a first chunk out of each prompt to fit
     the budget that is left;
  4. run the batch, then retire requests that have finished.
Invariant (§核心机制 2): the decodes are always in the batch and the batch
holds at most B tokens.  Request life cycle ("In-flight Batching", §调度状态机):
waiting -> prefill (chunked, repeated until the prompt is done) -> decode
(repeated) -> completed, with the pages freed at completion (§KV Cache 管理的
协同优化).  The last prefill chunk produces the first output token (§GPU / 系统
数据路径 ⑦), so a request enters decode with one generated token whose KV is
appended by its first decode step.

Readings where the pages are silent:
  * chunk size = min(prompt tokens left, budget left) ("fill the remaining
    budget"); ongoing chunks are also cut to the KV pages that can be had;
  * admission is first-come-first-served in arrival order and stops at the
    first request whose first chunk's pages cannot be allocated (no skipping);
  * pages are allocated only for the tokens scheduled this iteration, from the
    front of a FIFO free list; a finished request's pages go to its back in
    block-table order; there is no preemption: a decode that finds no free
    page is an error (OutOfPages);
  * if the running decodes alone exceed B they are all still scheduled (the
    decode half of the invariant wins), no prefill is added and the batch is
    flagged over_budget.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

WAITING, PREFILL, DECODE, DONE = "waiting", "prefill", "decode", "done"


class OutOfPages(RuntimeError):
    pass


@dataclass
class Request:
    rid: int
    prompt_len: int
    max_new: int
    phase: str = WAITING
    prefilled: int = 0
    generated: int = 0
    pages: list = field(default_factory=list)


@dataclass
class Row:
    rid: int
    kind: str            # "decode" | "prefill"
    q_len: int
    context_len: int     # tokens in cache after this step's append
    pages: list


@dataclass
class Batch:
    rows: list
    over_budget: bool

    @property
    def num_tokens(self):
        return sum(r.q_len for r in self.rows)

    def block_table(self, max_pages, fill=-1):
        return [r.pages + [fill] * (max_pages - len(r.pages)) for r in self.rows]


class StallFreeBuilder:
    """One scheduler instance: budget B tokens per iteration, a pool of
    `num_pages` pages of `page_size` tokens, sequences of at most
    `max_pages_per_seq` pages."""

    def __init__(self, budget, page_size, num_pages, max_pages_per_seq,
                 page_order=None):
        if budget < 1 or page_size < 1 or num_pages < 0 or max_pages_per_seq < 1:
            raise ValueError("bad builder parameters")
        self.budget = budget
        self.page_size = page_size
        self.max_pages_per_seq = max_pages_per_seq
        order = list(range(num_pages)) if page_order is None else list(page_order)
        if sorted(order) != list(range(num_pages)):
            raise ValueError("page_order must be a permutation of the pool")
        self.free = deque(order)
        self.waiting = deque()
        self.running = []          # admission order
        self.requests = {}
        self._pending = None

    # -- requests -----------------------------------------------------------
    def add_request(self, rid, prompt_len, max_new):
        if rid in self.requests:
            raise ValueError("duplicate request id")
        if prompt_len < 1 or max_new < 1:
            raise ValueError("prompt_len and max_new must be >= 1")
        longest = prompt_len + max_new - 1      # context of the last decode
        if -(-longest // self.page_size) > self.max_pages_per_seq:
            raise ValueError("request does not fit max_pages_per_seq")
        r = Request(rid, prompt_len, max_new)
        self.requests[rid] = r
        self.waiting.append(r)

    def _grow(self, r, n_tokens):
        """Make r's pages cover n_tokens tokens; False if pages ran out."""
        need = -(-n_tokens // self.page_size) - len(r.pages)
        if need > len(self.free):
            return False
        for _ in range(max(need, 0)):
            r.pages.append(self.free.popleft())
        return True

    # -- one iteration --------------------------------------------------------
    def step(self):
        """Form the next hybrid batch (None when there is nothing to run)."""
        if self._pending is not None:
            raise RuntimeError("complete() the previous batch first")
        rows, tokens = [], 0
        # 1. every running decode, one token each
        for r in self.running:
            if r.phase != DECODE:
                continue
            ctx = r.prompt_len + r.generated
            if not self._grow(r, ctx):
                raise OutOfPages(f"request {r.rid} needs a page for its decode")
            rows.append(Row(r.rid, "decode", 1, ctx, list(r.pages)))
            tokens += 1
        over_budget = tokens > self.budget
        # 2. continue unfinished prefills
        for r in self.running:
            if r.phase != PREFILL:
                continue
            left = self.budget - tokens
            if left <= 0:
                break
            c = min(r.prompt_len - r.prefilled, left)
            cap = (len(r.pages) + len(self.free)) * self.page_size - r.prefilled
            c = min(c, cap)
            if c <= 0:
                continue
            self._grow(r, r.prefilled + c)
            rows.append(Row(r.rid, "prefill", c, r.prefilled + c, list(r.pages)))
            tokens += c
        # 3. admit new requests, first-come-first-served
        while self.waiting and self.budget - tokens > 0:
            r = self.waiting[0]
            c = min(r.prompt_len, self.budget - tokens)
            if -(-c // self.page_size) > len(self.free):
                break
            self.waiting.popleft()
            r.phase = PREFILL
            self.running.append(r)
            self._grow(r, c)
            rows.append(Row(r.rid, "prefill", c, c, list(r.pages)))
            tokens += c
        if not rows:
            return None
        self._pending = Batch(rows, over_budget)
        return self._pending

    def complete(self, batch):
        """4. the batch ran: advance each request and retire finished ones."""
        if batch is not self._pending:
            raise RuntimeError("complete() must receive the batch step() returned")
        self._pending = None
        finished = []
        for row in batch.rows:
            r = self.requests[row.rid]
            if row.kind == "prefill":
                r.prefilled += row.q_len
                if r.prefilled == r.prompt_len:
                    r.phase = DECODE
                    r.generated = 1
            else:
                r.generated += 1
            if r.phase == DECODE and r.generated >= r.max_new:
                finished.append(r)
        for r in finished:
            r.phase = DONE
            self.running.remove(r)
            self.free.extend(r.pages)
            r.pages = []
        return [r.rid for r in finished]
