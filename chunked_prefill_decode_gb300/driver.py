"""Multi-iteration driver: synthetic request arrivals through the stall-free
builder and the attention step, with per-token latency statistics.

"Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
延迟权衡", §核心机制 2 and §GPU / 系统数据路径: every iteration the scheduler
forms one hybrid batch within a token budget, the GPU runs it, and each
running request advances (a decode emits a token; the last prefill chunk emits
the first one).  "Sarathi-Serve: Chunked Prefills for Stall-Free LLM
Inference", §Results and evidence: the quantity that matters is the
time-between-tokens (TBT) of running requests -- a decode that shares its
iteration with a whole long prefill stalls, one that shares it with a chunk
does not -- and the serving SLO is a multiple of an interference-free decode
iteration (strict about 5x, relaxed about 25x).

What this module does:
  * `poisson_requests` -- a seeded request stream: exponential inter-arrival
    times at a given rate, lognormal prompt and output lengths (the pages'
    medians, clipped), since the pages' traces are not available;
  * `run` -- drives the stream through the native builder (`hb.Builder`) and
    the library's append + attention on one device, advancing a clock by the
    measured device time of each iteration (CUDA events).  Only the attention
    layer is on this path, so an iteration's time is `layers` times that of
    one attention step (`layers` defaults to 1: attention of one layer).
    With `block` (a layer.BlockShape) the step runs a whole transformer
    block instead -- the linear layers on synthetic weights around the
    attention, all measured (`layer.HybridBlock`).  Without it, the linear
    layers can be added as a roofline estimate (`linear_params` > 0: the
    larger of 2 x params x tokens FLOPs at the dense bf16 peak and one read
    of the bf16 weights at the HBM rate) -- a model, not a measurement;
  * `latency_stats` -- TTFT and TBT percentiles from the token times;
  * `select_budget` -- the largest token budget whose P99 TBT stays within a
    multiple of the decode-only iteration time, from measured runs.

The step function is injectable (`step_time`), so the bookkeeping runs on the
CPU with a modelled cost in the tests; the real step needs a GPU.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass
class Request:
    rid: int
    arrival: float      # seconds
    prompt: int         # prompt tokens
    max_new: int        # output tokens (the first comes from the prefill)


def poisson_requests(rate: float, n: int, seed: int = 0, prompt_median: int = 1730,
                     output_median: int = 415, sigma: float = 0.6,
                     max_total: int = 8192) -> list[Request]:
    """n requests arriving as a Poisson process of `rate` per second, with
    lognormal(median, sigma) prompt and output lengths, prompt + output
    clipped to max_total (the openchat_sharegpt4 medians and truncation by
    default)."""
    if rate <= 0 or n < 0:
        raise ValueError("rate must be > 0 and n >= 0")
    rng = np.random.default_rng(seed)
    gaps = rng.exponential(1.0 / rate, size=n)
    t = np.cumsum(gaps)
    p = np.clip(np.rint(rng.lognormal(math.log(prompt_median), sigma, n)), 1, max_total - 1)
    o = np.rint(rng.lognormal(math.log(output_median), sigma, n))
    o = np.clip(o, 1, max_total - p)
    return [Request(i, float(t[i]), int(p[i]), int(o[i])) for i in range(n)]


@dataclass
class RunResult:
    budget: int
    iterations: int = 0
    clock: float = 0.0                      # seconds, end of the last iteration
    idle: float = 0.0                       # seconds with nothing to run
    iter_time: list = field(default_factory=list)      # seconds per iteration
    iter_tokens: list = field(default_factory=list)    # new tokens per iteration
    iter_decodes: list = field(default_factory=list)   # decode rows per iteration
    token_times: dict = field(default_factory=dict)    # rid -> [emission times]
    arrival: dict = field(default_factory=dict)        # rid -> arrival time
    unfinished: int = 0


def run(requests, budget: int, step_time, num_pages: int, max_pages_per_seq: int,
        page_size: int = 16, max_iterations: int = 100000, page_order=None) -> RunResult:
    """Drive `requests` through the library's builder.  `step_time(batch)`
    runs (or models) one iteration on the batch dict of `hb.Builder.step` and
    returns its duration in seconds.  Requests join when the clock has
    passed their arrival; an idle scheduler jumps to the next arrival."""
    from . import hb
    b = hb.Builder(budget, page_size, num_pages, max_pages_per_seq, page_order=page_order)
    pending = sorted(requests, key=lambda r: (r.arrival, r.rid))
    res = RunResult(budget)
    res.arrival = {r.rid: r.arrival for r in pending}
    prefill_left = {r.rid: r.prompt for r in pending}
    i = 0
    try:
        while res.iterations < max_iterations:
            while i < len(pending) and pending[i].arrival <= res.clock:
                r = pending[i]
                b.add_request(r.rid, r.prompt, r.max_new)
                i += 1
            batch = b.step()
            if batch is None:
                waiting, running, _ = b.counts()
                if i < len(pending) and waiting == 0 and running == 0:
                    res.idle += max(0.0, pending[i].arrival - res.clock)
                    res.clock = max(res.clock, pending[i].arrival)
                    continue
                if i >= len(pending) and waiting == 0 and running == 0:
                    break
                # requests wait for pages that no running request will free
                raise RuntimeError("builder stalled: waiting requests cannot be admitted")
            dt = float(step_time(batch))
            res.clock += dt
            res.iterations += 1
            res.iter_time.append(dt)
            res.iter_tokens.append(int(batch["q_len"].sum()))
            res.iter_decodes.append(int((batch["kind"] == 0).sum()))
            # tokens emitted at the end of this iteration: one per decode row,
            # and the first token of every prompt whose last chunk ran
            for rid, kind, ql in zip(batch["ids"].tolist(), batch["kind"].tolist(),
                                     batch["q_len"].tolist()):
                if kind == 0:
                    res.token_times.setdefault(rid, []).append(res.clock)
                else:
                    prefill_left[rid] -= ql
                    if prefill_left[rid] == 0:
                        res.token_times.setdefault(rid, []).append(res.clock)
            b.complete()
        waiting, running, _ = b.counts()
        res.unfinished = waiting + running + (len(pending) - i)
    finally:
        b.close()
    return res


def latency_stats(res: RunResult) -> dict:
    """TTFT (arrival -> first token) and TBT (gaps between a request's
    consecutive tokens) percentiles in milliseconds, output tokens per second."""
    ttft, tbt = [], []
    n_tok = 0
    for rid, times in res.token_times.items():
        n_tok += len(times)
        ttft.append(times[0] - res.arrival[rid])
        tbt.extend(np.diff(times).tolist())

    def pct(x, q):
        return float(np.percentile(x, q) * 1e3) if len(x) else None
    return {
        "budget": res.budget, "iterations": res.iterations, "requests": len(res.token_times),
        "unfinished": res.unfinished, "output_tokens": n_tok,
        "output_tokens_per_s": n_tok / res.clock if res.clock > 0 else None,
        "ttft_ms_p50": pct(ttft, 50), "ttft_ms_p99": pct(ttft, 99),
        "tbt_ms_p50": pct(tbt, 50), "tbt_ms_p90": pct(tbt, 90), "tbt_ms_p99": pct(tbt, 99),
        "tbt_ms_max": float(max(tbt) * 1e3) if tbt else None,
        "iter_ms_max": float(max(res.iter_time) * 1e3) if res.iter_time else None,
        "iter_tokens_max": max(res.iter_tokens) if res.iter_tokens else 0,
    }


def select_budget(stats_by_budget: dict, decode_iter_ms: float, slo_multiple: float = 5.0):
    """The largest budget whose P99 TBT is within slo_multiple x the
    decode-only iteration time, or None.  stats_by_budget: budget ->
    latency_stats dict."""
    limit = slo_multiple * decode_iter_ms
    ok = [b for b, s in stats_by_budget.items()
          if s.get("tbt_ms_p99") is not None and s["tbt_ms_p99"] <= limit]
    return max(ok) if ok else None


class GpuStep:
    """The library's append + plan + attention for one batch on one device,
    timed with CUDA events; K/V pools persist across iterations (the values
    of q and the new K/V are random -- only the time is used)."""

    def __init__(self, num_pages, num_q_heads=32, num_kv_heads=8, head_dim=128,
                 page_size=16, layers=1, seed=0, device="cuda", sliding_window=0,
                 linear_params=0.0, peak_tflops=None, hbm_gbs=None, block=None):
        import torch
        from . import hb
        self.torch, self.hb = torch, hb
        self.dev = torch.device(device)
        self.shape = (num_q_heads, num_kv_heads, head_dim, page_size)
        self.layers = layers
        self.window = sliding_window
        if linear_params > 0 and (not peak_tflops or not hbm_gbs):
            raise ValueError("the linear-layer model needs peak_tflops and hbm_gbs")
        self.linear_params = linear_params
        self.peak_tflops, self.hbm_gbs = peak_tflops, hbm_gbs
        self.block = None
        if block is not None:
            from .layer import HybridBlock
            if (block.num_q_heads, block.num_kv_heads, block.head_dim, block.page_size) != \
                    (num_q_heads, num_kv_heads, head_dim, page_size):
                raise ValueError("block shape and attention shape differ")
            self.block = HybridBlock(block, seed=seed, device=device)
        self.num_pages = num_pages
        g = torch.Generator(device=self.dev).manual_seed(seed)
        pool = (num_pages, page_size, num_kv_heads, head_dim)
        self.k_pool = torch.randn(pool, generator=g, device=self.dev).to(torch.bfloat16)
        self.v_pool = torch.randn(pool, generator=g, device=self.dev).to(torch.bfloat16)
        self.gen = g
        self.sms = torch.cuda.get_device_properties(self.dev).multi_processor_count
        self.scale = 1.0 / math.sqrt(head_dim)
        self.ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        self.plan = None
        self.ws = None

    def __call__(self, batch) -> float:
        from .device import device_batch
        torch = self.torch
        hq, hkv, d, P = self.shape
        ql, cl, bt = batch["q_len"], batch["context_len"], batch["block_table"]
        T = int(ql.sum())
        q = torch.randn(T, hq, d, generator=self.gen, device=self.dev).to(torch.bfloat16)
        kn = torch.randn(T, hkv, d, generator=self.gen, device=self.dev).to(torch.bfloat16)
        vn = torch.randn(T, hkv, d, generator=self.gen, device=self.dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        db = device_batch(ql, cl, bt, self.num_pages, hq, hkv, d, P, self.dev,
                          sliding_window=self.window)
        self.plan, self.ws = self.hb.hb_plan(db.batch, db.q_len, db.context_len, self.sms,
                                             workspace=self.ws, plan=self.plan)
        if self.block is not None:
            blk = self.block
            blk._plan, blk._ws = self.plan, self.ws
            x = torch.randn(T, blk.shape.hidden, generator=self.gen,
                            device=self.dev).to(torch.bfloat16)
            torch.cuda.synchronize(self.dev)
            e0, e1 = self.ev
            e0.record()
            blk.forward(x, db, self.k_pool, self.v_pool, plan=False)
            e1.record()
            torch.cuda.synchronize(self.dev)
            self.hb.hb_check()
            return self.layers * e0.elapsed_time(e1) * 1e-3
        torch.cuda.synchronize(self.dev)
        e0, e1 = self.ev
        e0.record()
        self.hb.hb_kv_append(db.batch, kn, vn, self.k_pool, self.v_pool)
        self.hb.hb_attention_new_kv(db.batch, self.plan, q, kn, vn, self.k_pool, self.v_pool,
                                    self.scale, out, self.ws)
        e1.record()
        torch.cuda.synchronize(self.dev)
        self.hb.hb_check()
        return self.layers * e0.elapsed_time(e1) * 1e-3 + self.linear_time(T)

    def linear_time(self, tokens: int) -> float:
        """Roofline estimate (seconds) of the linear layers for `tokens` new
        tokens; 0 unless linear_params was given."""
        if self.linear_params <= 0:
            return 0.0
        flops = 2.0 * self.linear_params * tokens
        weight_bytes = 2.0 * self.linear_params
        return max(flops / (self.peak_tflops * 1e12), weight_bytes / (self.hbm_gbs * 1e9))


def decode_only_iteration_ms(step: GpuStep, n_rows: int, context: int, max_pages_per_seq: int,
                             reps: int = 5) -> float:
    """Median time of an interference-free decode iteration: n_rows decode
    rows at the given context, nothing else in the batch."""
    P = step.shape[3]
    npg = -(-context // P)
    if n_rows * npg > step.num_pages:
        raise ValueError("pool too small for the decode-only batch")
    bt = np.full((n_rows, max_pages_per_seq), -1, np.int32)
    for r in range(n_rows):
        bt[r, :npg] = np.arange(r * npg, (r + 1) * npg)
    batch = {"q_len": np.ones(n_rows, np.int32),
             "context_len": np.full(n_rows, context, np.int32), "block_table": bt}
    times = sorted(step(batch) for _ in range(reps))
    return times[len(times) // 2] * 1e3


def main(argv=None):
    import argparse
    import json
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--rate", type=float, default=6.0, help="requests per second")
    ap.add_argument("--requests", type=int, default=200)
    ap.add_argument("--budgets", default="256,512,1024,2048,8192",
                    help="token budgets to run (8192: whole prompts in one iteration)")
    ap.add_argument("--layers", type=int, default=32,
                    help="attention layers per iteration (Mistral-7B: 32)")
    ap.add_argument("--num-pages", type=int, default=24000)
    ap.add_argument("--slo", type=float, default=5.0,
                    help="P99 TBT limit as a multiple of the decode-only iteration")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--block", choices=["none", "mistral"], default="none",
                    help="run a whole Mistral-7B-shaped block per layer (measured linear "
                         "layers on synthetic weights) instead of attention alone")
    ap.add_argument("--linear-params", type=float, default=0.0,
                    help="add a roofline estimate of linear layers with this many "
                         "bf16 parameters (Mistral-7B: about 7.1e9); 0 = attention only")
    ap.add_argument("--peak-tflops", type=float, default=None,
                    help="dense bf16 peak for the linear-layer estimate")
    ap.add_argument("--hbm-gbs", type=float, default=None,
                    help="HBM bandwidth for the linear-layer estimate")
    args = ap.parse_args(argv)
    reqs = poisson_requests(args.rate, args.requests, seed=args.seed)
    maxp = 8192 // 16
    block = None
    if args.block == "mistral":
        from .layer import MISTRAL_7B
        block = MISTRAL_7B
    step = GpuStep(args.num_pages, layers=args.layers, seed=args.seed,
                   linear_params=args.linear_params, peak_tflops=args.peak_tflops,
                   hbm_gbs=args.hbm_gbs, block=block)
    base_ms = decode_only_iteration_ms(step, 32, 2048, maxp)
    stats = {}
    for bud in [int(x) for x in args.budgets.split(",")]:
        res = run(reqs, bud, step, args.num_pages, maxp)
        stats[bud] = latency_stats(res)
        print(json.dumps({"driver": "poisson", "rate": args.rate, "layers": args.layers,
                          "block": args.block, "linear_params_modelled": args.linear_params,
                          **stats[bud]}), flush=True)
    print(json.dumps({"decode_only_iter_ms": base_ms, "slo_multiple": args.slo,
                      "selected_budget": select_budget(stats, base_ms, args.slo)}), flush=True)


if __name__ == "__main__":
    main()
