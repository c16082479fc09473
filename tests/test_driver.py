"""The multi-iteration driver: request streams, token-time bookkeeping over the
native builder, latency statistics and budget selection.  CPU tests use a
modelled iteration cost; the GPU test runs the real append + attention."""
import math

import numpy as np
import pytest

from chunked_prefill_decode_gb300 import driver


def linear_cost(base_s=1e-3, per_token_s=2e-5):
    """Modelled iteration time: a fixed part plus a part per new token."""
    return lambda batch: base_s + per_token_s * float(batch["q_len"].sum())


def test_poisson_stream_statistics():
    reqs = driver.poisson_requests(rate=10.0, n=4000, seed=3)
    gaps = np.diff([0.0] + [r.arrival for r in reqs])
    assert abs(gaps.mean() - 0.1) < 0.01                     # mean inter-arrival 1 / rate
    assert abs(np.std(gaps) / gaps.mean() - 1.0) < 0.1       # exponential: CV = 1
    assert abs(np.median([r.prompt for r in reqs]) - 1730) < 120
    assert abs(np.median([r.max_new for r in reqs]) - 415) < 40
    assert all(1 <= r.prompt and 1 <= r.max_new and r.prompt + r.max_new <= 8192 for r in reqs)
    assert [r.arrival for r in reqs] == sorted(r.arrival for r in reqs)


def test_every_request_gets_all_its_tokens_in_order():
    reqs = driver.poisson_requests(rate=50.0, n=40, seed=1, prompt_median=300,
                                   output_median=20, max_total=1024)
    res = driver.run(reqs, 128, linear_cost(), num_pages=3000, max_pages_per_seq=64)
    assert res.unfinished == 0
    for r in reqs:
        t = res.token_times[r.rid]
        assert len(t) == r.max_new                 # the prefill's token + max_new - 1 decodes
        assert t[0] > r.arrival and all(np.diff(t) > 0)
    assert math.isclose(res.clock, sum(res.iter_time) + res.idle)
    assert max(res.iter_tokens) <= 128 or max(res.iter_decodes) > 128


def test_idle_scheduler_jumps_to_the_next_arrival():
    reqs = [driver.Request(0, 0.0, 20, 3), driver.Request(1, 100.0, 20, 3)]
    res = driver.run(reqs, 64, linear_cost(), num_pages=100, max_pages_per_seq=8)
    assert res.token_times[1][0] > 100.0 and res.token_times[0][-1] < 1.0
    assert res.iterations == 6                      # 1 prefill + 2 decodes, twice


def test_chunking_bounds_the_time_between_tokens():
    """With an iteration cost that grows with its tokens, admitting whole
    prompts (a large budget) stretches the gaps between a running request's
    tokens; a small budget keeps every iteration, and so every gap, short."""
    reqs = driver.poisson_requests(rate=20.0, n=60, seed=2, prompt_median=1500,
                                   output_median=60, max_total=4096)
    stats = {}
    for bud in (256, 8192):
        res = driver.run(reqs, bud, linear_cost(), num_pages=20000, max_pages_per_seq=256)
        assert res.unfinished == 0
        stats[bud] = driver.latency_stats(res)
    assert stats[256]["iter_tokens_max"] <= 256 + 64
    assert stats[256]["tbt_ms_max"] < stats[8192]["tbt_ms_max"] / 3
    assert stats[256]["tbt_ms_p99"] < stats[8192]["tbt_ms_p99"]
    # the cost: first tokens come later with small chunks
    assert stats[256]["ttft_ms_p50"] > stats[8192]["ttft_ms_p50"]


def test_latency_stats_by_hand():
    res = driver.RunResult(budget=8, clock=1.0, iter_time=[0.5, 0.5], iter_tokens=[3, 1])
    res.arrival = {7: 0.0, 9: 0.25}
    res.token_times = {7: [0.5, 0.75, 1.0], 9: [0.5]}
    s = driver.latency_stats(res)
    assert s["output_tokens"] == 4 and s["output_tokens_per_s"] == 4.0
    assert s["tbt_ms_max"] == 250.0 and s["tbt_ms_p50"] == 250.0
    assert s["ttft_ms_p50"] == pytest.approx(375.0)


def test_select_budget():
    stats = {256: {"tbt_ms_p99": 4.0}, 512: {"tbt_ms_p99": 9.0}, 1024: {"tbt_ms_p99": 11.0},
             2048: {"tbt_ms_p99": 30.0}}
    assert driver.select_budget(stats, decode_iter_ms=2.0, slo_multiple=5.0) == 512
    assert driver.select_budget(stats, decode_iter_ms=2.0, slo_multiple=25.0) == 2048
    assert driver.select_budget(stats, decode_iter_ms=0.5, slo_multiple=5.0) is None


@pytest.mark.gpu
def test_driver_on_the_gpu():
    """A short stream through the real append + attention: all requests finish
    with all their tokens, and the decode-only iteration is timed.  (With
    attention alone a prefill chunk costs little next to the decode stream,
    so no ordering of the budgets' gaps is asserted here; see the block test.)"""
    reqs = driver.poisson_requests(rate=400.0, n=24, seed=5, prompt_median=1200,
                                   output_median=12, max_total=4096)
    step = driver.GpuStep(num_pages=8000, layers=1, seed=5)
    for bud in (256, 8192):
        res = driver.run(reqs, bud, step, num_pages=8000, max_pages_per_seq=256)
        assert res.unfinished == 0
        assert all(len(res.token_times[r.rid]) == r.max_new for r in reqs)
        assert min(res.iter_time) > 0
    assert driver.decode_only_iteration_ms(step, 8, 1024, 256) > 0


def test_linear_layer_roofline_estimate():
    """2 P T FLOPs at the bf16 peak, or one read of the 2 P weight bytes at the
    HBM rate, whichever is longer (decodes are weight-bound, prefills
    compute-bound)."""
    s = driver.GpuStep.__new__(driver.GpuStep)
    s.linear_params, s.peak_tflops, s.hbm_gbs = 7.0e9, 2000.0, 7000.0
    assert s.linear_time(1) == pytest.approx(2 * 7.0e9 / 7000e9)          # 2 ms, weights
    assert s.linear_time(4096) == pytest.approx(2 * 7.0e9 * 4096 / 2000e12)
    crossover = 2000e12 / 7000e9                                         # tokens
    assert s.linear_time(int(crossover) - 1) == pytest.approx(2e-3)
    s.linear_params = 0.0
    assert s.linear_time(4096) == 0.0


@pytest.mark.gpu
def test_driver_with_whole_blocks_on_the_gpu():
    """With whole transformer blocks per iteration (measured linear layers
    around the attention step), an iteration's time grows with its tokens, so
    admitting whole prompts stretches the worst gap between a running
    request's tokens beyond what a 256-token budget allows.  (Mistral-7B-sized
    blocks: an 8192-token iteration then holds milliseconds of GPU work, well
    above the host's share of an iteration, which a smaller block would not.)"""
    from chunked_prefill_decode_gb300.layer import BlockShape
    reqs = driver.poisson_requests(rate=2000.0, n=12, seed=6, prompt_median=1500,
                                   output_median=8, max_total=4096)
    blk = BlockShape(hidden=4096, num_q_heads=32, num_kv_heads=8, head_dim=128, ffn=14336)
    step = driver.GpuStep(num_pages=6000, layers=2, seed=6, block=blk)
    worst = {}
    for bud in (256, 8192):
        res = driver.run(reqs, bud, step, num_pages=6000, max_pages_per_seq=256)
        assert res.unfinished == 0 and min(res.iter_time) > 0
        assert all(len(res.token_times[r.rid]) == r.max_new for r in reqs)
        worst[bud] = driver.latency_stats(res)["tbt_ms_max"]
    assert worst[256] < worst[8192]
