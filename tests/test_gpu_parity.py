"""CUDA path against the fp64 oracle, through the C ABI (GB300).

Small batches are compared element by element; full-size workloads on the
rows the oracle can afford (every decode row of a sample of sequences, a
sample of chunk tokens).  Bars: KV append bit-exact, attention max-abs <= 1e-2
and mean-abs <= 1e-3 (bf16 inputs, fp32 accumulation).
"""
import math

import numpy as np
import pytest
import torch

from _gpu import MAX_ABS, MEAN_ABS, bits, compact_layout, compare, gpu_step, oracle_step, sms
from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from chunked_prefill_decode_gb300.workloads import Shape, layout_from_rows

pytestmark = pytest.mark.gpu


def _full_check(layout, seed=0, scale=None, repeats=1):
    ten = workloads.make_tensors(layout, seed)
    kc, vc, out = gpu_step(layout, ten, scale=scale, repeats=repeats)
    kp, vp, ref = oracle_step(layout, ten, scale=scale)
    assert np.array_equal(bits(kc), kp), "K append differs"
    assert np.array_equal(bits(vc), vp), "V append differs"
    return compare(out, ref)


def test_tiny_workload():
    _full_check(workloads.tiny(0))


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_tiny_workload_seeds(seed):
    _full_check(workloads.tiny(seed), seed=seed)


def test_repeated_attention_reuses_plan():
    # counters in the workspace must reset themselves between launches
    lay = layout_from_rows(Shape(32, 8, 128), [(1, 3000)] * 6 + [(1, 700), (40, 300)], 5)
    _full_check(lay, seed=5, repeats=4)


@pytest.mark.parametrize("rows", [
    [(1, 1)], [(1, 16)], [(1, 17)], [(1, 128)], [(1, 129)], [(1, 2047)],
    [(2, 2)], [(15, 15)], [(16, 16)], [(17, 17)], [(127, 127)], [(128, 128)],
    [(129, 129)], [(257, 257)], [(64, 1000)], [(100, 1029)], [(33, 4096)],
    [(1, 50), (1, 700), (5, 37), (130, 700), (1, 3)],
])
@pytest.mark.parametrize("geom", [(8, 8, 64), (32, 8, 128), (56, 8, 128)])
def test_edge_rows(rows, geom):
    hq, hkv, d = geom
    _full_check(layout_from_rows(Shape(hq, hkv, d), rows, 11), seed=11)


@pytest.mark.parametrize("geom", [(4, 4, 128), (16, 2, 64), (64, 16, 128), (32, 32, 128), (16, 1, 128),
                                  (8, 1, 64), (128, 8, 128)])
def test_other_head_geometries(geom):
    hq, hkv, d = geom
    rows = [(1, 200), (1, 37), (24, 90), (1, 1000)]
    _full_check(layout_from_rows(Shape(hq, hkv, d), rows, 12), seed=12)


@pytest.mark.parametrize("geom,rows,window", [
    ((32, 8, 128), [(512, 1024)], 0),                    # chunk at offset 512: page-aligned
    ((32, 8, 128), [(257, 1000)], 0),                    # offset 743: its first page straddles
    ((32, 8, 128), [(100, 100)], 0),                     # offset 0: every page is new
    ((56, 8, 128), [(1, 3000)] * 4 + [(2016, 7059)], 0),  # pairs, offset 5043
    ((56, 8, 128), [(1, 2000)] * 2 + [(48, 6048)], 0),
    ((8, 8, 64), [(300, 3000), (1, 50), (33, 33)], 0),
    ((16, 1, 128), [(300, 9000)], 0),                    # split pieces
    ((32, 8, 128), [(448, 4000), (1, 3000)], 1024),      # sliding window
    ((32, 8, 128), [(130, 700), (5, 37), (1, 3)], 7),
])
def test_attention_with_new_rows(geom, rows, window):
    """hb_attention_new_kv reads the chunks' pages of new tokens from k_new /
    v_new instead of the caches: with the same plan the products are the same
    on the same bf16 values, so the output equals hb_attention's bit for bit,
    and it meets the oracle's bars."""
    hq, hkv, d = geom
    lay = layout_from_rows(Shape(hq, hkv, d, sliding_window=window), rows, 21)
    ten = workloads.make_tensors(lay, 21)
    _, _, out_cache = gpu_step(lay, ten)
    kc, vc, out_new = gpu_step(lay, ten, new_kv=True)
    assert torch.equal(out_cache.view(torch.int16), out_new.view(torch.int16))
    kp, vp, ref = oracle_step(lay, ten)
    assert np.array_equal(bits(kc), kp) and np.array_equal(bits(vc), vp)
    compare(out_new, ref)


@pytest.mark.parametrize("geom,rows", [
    ((32, 8, 128), [(64, 4160)]),
    ((32, 8, 128), [(1, 2048)] * 8 + [(96, 6000)]),
    ((8, 8, 64), [(100, 3000)]),
    ((56, 8, 128), [(1, 5000), (40, 5040)]),
    ((16, 1, 128), [(300, 9000)]),
])
def test_split_key_ranges(geom, rows):
    """Chunks with too few query tiles to fill the SMs, at long offsets: the
    plan cuts each tile's key range into pieces that the last piece to finish
    merges.  Three launches on one plan also check that the merge counters
    reset themselves."""
    from _hbutil import host_batch
    hq, hkv, d = geom
    hb = lib()
    b, ql, cl = host_batch(hb, rows, hq=hq, hkv=hkv, d=d)
    plan, _ = hb.hb_plan(b, ql, cl, sms(), upload=False)
    assert hb.plan_header(plan)["num_chunk_merges"] > 0
    _full_check(layout_from_rows(Shape(hq, hkv, d), rows, 14), seed=14, repeats=3)


@pytest.mark.parametrize("geom,rows,window", [
    ((32, 8, 128), [(512, 8192)], 0),
    ((56, 8, 128), [(252, 8000)], 0),
    ((32, 8, 128), [(1, 2048)] * 8 + [(512, 7000)], 0),
    ((16, 1, 128), [(600, 9000)], 0),
    ((32, 8, 128), [(200, 5000), (300, 6000)], 0),
    ((32, 8, 128), [(256, 8192)], 3000),
])
def test_split_pairs(geom, rows, window):
    """Pairs of query tiles whose key range is cut into pieces (with single
    tiles split alongside in the mixed batch): each piece publishes both
    tiles' partial states, a tile past its own last key publishes none, and
    the last piece merges them.  Sampled rows of every chunk against the
    oracle, three launches on one plan."""
    from _hbutil import host_batch
    hq, hkv, d = geom
    hb = lib()
    b, ql, cl = host_batch(hb, rows, hq=hq, hkv=hkv, d=d, window=window)
    plan, _ = hb.hb_plan(b, ql, cl, sms(), upload=False)
    tpt = hb.plan_header(plan)["chunk_tokens_per_tile"]
    _, chk, _ = hb.plan_items(plan)
    assert ((chk[:, 3] > tpt) & (chk[:, 10] > 1)).any()
    lay = layout_from_rows(Shape(hq, hkv, d, sliding_window=window), rows, 19)
    _full_size(None, seed=19, lay=lay, repeats=3)


@pytest.mark.parametrize("rows", [
    [(2, 2)], [(3, 3)], [(17, 17)], [(33, 40)], [(100, 100)], [(130, 1000)],
    [(255, 256)], [(257, 300)], [(1, 129), (64, 4160), (1, 7)], [(600, 1200), (1, 50), (9, 9)],
])
@pytest.mark.parametrize("geom", [(32, 8, 128), (56, 8, 128), (8, 8, 64)])
def test_fresh_and_short_chunks(rows, geom):
    """Chunks of 2 .. 600 tokens at offsets 0 .. 4096: the first tokens of a
    prompt see few keys, so their output leans on a few softmax weights (such
    items carry P in two bf16 terms); odd key-tile counts, short or empty
    second tiles, last pages with unwritten slots."""
    hq, hkv, d = geom
    _full_check(layout_from_rows(Shape(hq, hkv, d), rows, 31), seed=31)


@pytest.mark.parametrize("seed", range(6))
def test_random_batches_with_short_windows(seed):
    """Random hybrid batches whose windows (1 .. 300 keys) or fresh chunks
    leave every chunk row few keys."""
    rng = np.random.default_rng(3000 + seed)
    hq, hkv, d = [(32, 8, 128), (56, 8, 128), (64, 16, 128), (16, 1, 128), (8, 8, 64),
                  (56, 8, 128)][seed]
    rows = [(1, int(rng.integers(1, 2500))) for _ in range(int(rng.integers(0, 12)))]
    for _ in range(int(rng.integers(1, 3))):
        q = int(rng.integers(2, 400))
        rows.append((q, q + int(rng.integers(0, 1500))))
    rng.shuffle(rows)
    window = int(rng.choice([0, 0, 5, 300])) if seed < 4 else [5, 1][seed - 4]
    _full_check(layout_from_rows(Shape(hq, hkv, d, sliding_window=window),
                                 [tuple(r) for r in rows], 3000 + seed), seed=seed)


WINDOW_ROWS = [(1, 1), (1, 17), (1, 700), (1, 3000), (5, 37), (130, 700), (64, 4160),
               (257, 2000), (1, 129)]


@pytest.mark.parametrize("window", [1, 7, 16, 100, 1000, 5000])
@pytest.mark.parametrize("geom", [(8, 8, 64), (32, 8, 128), (56, 8, 128)])
def test_sliding_window(window, geom):
    """Sliding-window attention: decode rows start their page range at the
    window, chunk tiles their key range, and both mask the window's edge."""
    hq, hkv, d = geom
    _full_check(layout_from_rows(Shape(hq, hkv, d, sliding_window=window), WINDOW_ROWS, 15),
                seed=15, repeats=2)


def _round_bf16(x):
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("seed", [15, 17])
@pytest.mark.parametrize("case", ["w1", "w7", "w16", "w100", "fresh17", "fresh127"])
@pytest.mark.parametrize("geom", [(8, 8, 64), (32, 8, 128), (56, 8, 128)])
def test_error_beyond_output_rounding_keeps_headroom(case, geom, seed):
    """The bf16 output cannot be closer to the fp64 answer than that answer's
    own bf16 rounding, which alone reaches half an ulp: 0.0078 just above
    |o| = 2, 78 % of the max-abs bound (and ~55 % of the mean-abs bound on
    rows with few keys).  What the kernel adds on top of that rounding (the
    bf16 softmax weights, the fp32 sums) stays at or below 80 % of both
    bounds, on short windows and fresh prefills, where few keys per row make
    it largest."""
    hq, hkv, d = geom
    if case.startswith("w"):
        lay = layout_from_rows(Shape(hq, hkv, d, sliding_window=int(case[1:])), WINDOW_ROWS, seed)
    else:
        n = int(case[5:])
        lay = layout_from_rows(Shape(hq, hkv, d), [(n, n), (1, 50), (1, 3)], seed)
    ten = workloads.make_tensors(lay, seed)
    kc, vc, out = gpu_step(lay, ten)
    kp, vp, ref = oracle_step(lay, ten)
    assert np.array_equal(bits(kc), kp) and np.array_equal(bits(vc), vp)
    compare(out, ref)
    got = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    floor = np.abs(_round_bf16(ref) - ref)        # the exact answer's own rounding
    assert (err - floor).max() <= 0.8 * MAX_ABS, (err - floor).max()
    assert err.mean() - floor.mean() <= 0.8 * MEAN_ABS, (err.mean(), floor.mean())


@pytest.mark.parametrize("window", [16, 100, 1000])
def test_sliding_window_never_reads_pages_below_it(window):
    """Block-table entries of pages below every window of their row are set
    to -1 (as a cache that has freed them would): no index error, same result."""
    lay = layout_from_rows(Shape(32, 8, 128, sliding_window=window), WINDOW_ROWS, 16)
    ten = workloads.make_tensors(lay, 16)
    P = lay.shape.page_size
    for s in range(lay.num_seqs):
        lowest = int(lay.context_len[s] - lay.q_len[s]) - window + 1
        n_below = max(0, lowest) // P
        lay.block_table[s, :n_below] = -1
    kc, vc, out = gpu_step(lay, ten)          # hb_check raises on an index error
    _, _, ref = oracle_step(lay, ten)
    compare(out, ref)


@pytest.mark.parametrize("n_seqs", [6143, 6144, 7000])
def test_append_with_many_sequences(n_seqs):
    """Up to 6143 sequences the append kernel stages cu_q_len and
    context_len in shared memory; beyond, it searches them in global memory.
    Both copies are bit-exact, and attention over the batch still holds on a
    sample of its rows."""
    rng = np.random.default_rng(n_seqs)
    rows = [(1, int(c)) for c in rng.integers(1, 40, size=n_seqs - 2)] + [(5, 9), (33, 70)]
    lay = layout_from_rows(Shape(8, 1, 64), rows, 18)
    ten = workloads.make_tensors(lay, 18)
    kc, vc, out = gpu_step(lay, ten)
    sample = sorted(rng.choice(lay.total_q, size=200, replace=False).tolist())
    kp, vp, ref = oracle_step(lay, ten, tokens=sample)
    assert np.array_equal(bits(kc), kp), "K append differs"
    assert np.array_equal(bits(vc), vp), "V append differs"
    compare(out, ref, tokens=sample)


def test_several_chunks_and_decodes():
    rows = [(1, 900)] * 7 + [(200, 456), (57, 57), (300, 2000), (1, 5)]
    _full_check(layout_from_rows(Shape(32, 8, 128), rows, 13), seed=13)


def test_constant_v_returns_v_exactly():
    lay = layout_from_rows(Shape(32, 8, 128), [(1, 1500), (1, 40), (150, 400)], 14)
    ten = workloads.make_tensors(lay, 14)
    hkv, d = 8, 128
    c = torch.randn(hkv, d).to(torch.bfloat16)
    ten.v_new[:] = c
    keep = torch.from_numpy(workloads.cached_slot_mask(lay))
    ten.v_cache[keep] = c
    _, _, out = gpu_step(lay, ten)
    expect = c.repeat_interleave(4, dim=0)
    assert torch.equal(out.cpu(), expect[None].expand_as(out.cpu()))


def test_chunked_prefill_equals_unchunked_on_gpu():
    """A 700-token prompt prefilled in chunks of 1, 100, 128, 257 and at once:
    every chunking matches the oracle, and they agree with each other."""
    L, sh = 700, Shape(32, 8, 128)
    g = torch.Generator().manual_seed(15)
    q = torch.randn(L, 32, 128, generator=g).to(torch.bfloat16)
    kn = torch.randn(L, 8, 128, generator=g).to(torch.bfloat16)
    vn = torch.randn(L, 8, 128, generator=g).to(torch.bfloat16)
    base = layout_from_rows(sh, [(L, L)], 15)
    pool_k = torch.zeros(base.num_pages, 16, 8, 128, dtype=torch.bfloat16)
    pool_v = torch.zeros_like(pool_k)
    outs = {}
    for c in (L, 1, 100, 128, 257):
        kp, vp = pool_k.clone(), pool_v.clone()
        res = []
        for start in range(0, L, c) if c > 1 else range(0, 40):  # chunk 1: first 40 tokens
            n = min(c, L - start)
            lay = workloads.BatchLayout(sh, np.array([n], np.int32),
                                        np.array([start + n], np.int32),
                                        base.block_table, base.num_pages)
            ten = workloads.BatchTensors(q[start:start + n].clone(), kn[start:start + n].clone(),
                                         vn[start:start + n].clone(), kp, vp)
            kc, vc, out = gpu_step(lay, ten)
            _, _, ref = oracle_step(lay, ten)
            compare(out, ref)
            kp, vp = kc.cpu(), vc.cpu()
            res.append(out.float().cpu())
        outs[c] = torch.cat(res)
    for c in (100, 128, 257):
        assert (outs[c] - outs[L]).abs().max().item() <= 2 * MAX_ABS
    assert (outs[1] - outs[L][:40]).abs().max().item() <= 2 * MAX_ABS


def test_device_index_error_is_reported():
    hb = lib()
    lay = layout_from_rows(Shape(8, 8, 64), [(1, 40), (20, 50)], 16)
    ten = workloads.make_tensors(lay, 16)
    lay.block_table[0, 1] = lay.num_pages + 5      # out of range
    lay.block_table[1, 0] = -3
    gpu_step(lay, ten, check=False)
    with pytest.raises(hb.HbError) as e:
        hb.hb_check()
    assert e.value.status == 6
    hb.hb_check()   # the word was cleared


def test_timing_and_launch_count():
    hb = lib()
    lay = workloads.tiny(0)
    ten = workloads.make_tensors(lay, 0)
    n0 = hb.hb_launch_count()
    hb.hb_timing_enable(True)
    gpu_step(lay, ten)
    t = hb.hb_timing_read()
    hb.hb_timing_enable(False)
    assert hb.hb_launch_count() - n0 == 2
    for name in ("kv_append", "attention"):
        assert t[name][1] == 1 and t[name][0] > 0
    # sampling: records survive a pause and a resume adds to them
    hb.hb_timing_enable(True)
    gpu_step(lay, ten)
    hb.hb_timing_enable(False)
    gpu_step(lay, ten)
    hb.hb_timing_enable(True, keep=True)
    gpu_step(lay, ten)
    hb.hb_timing_enable(False)
    t = hb.hb_timing_read()
    for name in ("kv_append", "attention"):
        assert t[name][1] == 2


# ---------------------------------------------------------------- full size
def _full_size(name, n_seq_sample=6, n_chunk_tok=48, seed=None, lay=None, repeats=1):
    if lay is None:
        lay = workloads.WORKLOADS[name]()
    seed = {"mistral_b512": 1, "mistral_b512_window": 1, "yi_b2048": 2, "yi_b2048_o5043": 2,
            "decode_only": 3}.get(name, 0) if seed is None else seed
    ten = workloads.make_tensors(lay, seed, device="cuda")
    kc, vc, out = gpu_step(lay, ten, repeats=repeats)
    rng = np.random.default_rng(seed)
    dec = [s for s in range(lay.num_seqs) if lay.q_len[s] == 1]
    chk = [s for s in range(lay.num_seqs) if lay.q_len[s] > 1]
    # append: bit-exact at every written slot, untouched elsewhere (device)
    cu = lay.cu_q_len
    P = lay.shape.page_size
    pos = np.concatenate([np.arange(lay.context_len[s] - lay.q_len[s], lay.context_len[s])
                          for s in range(lay.num_seqs)])
    seq_of = np.repeat(np.arange(lay.num_seqs), lay.q_len)
    pages = lay.block_table[seq_of, pos // P]
    slots = pos % P
    pg = torch.from_numpy(pages.astype(np.int64)).cuda()
    sl = torch.from_numpy(slots.astype(np.int64)).cuda()
    assert torch.equal(kc[pg, sl].view(torch.int16), ten.k_new.view(torch.int16))
    assert torch.equal(vc[pg, sl].view(torch.int16), ten.v_new.view(torch.int16))
    written = torch.zeros(kc.shape[:2], dtype=torch.bool, device="cuda")
    written[pg, sl] = True
    assert torch.equal(kc.view(torch.int16)[~written], ten.k_cache.view(torch.int16)[~written])
    assert torch.equal(vc.view(torch.int16)[~written], ten.v_cache.view(torch.int16)[~written])
    # attention on sampled sequences
    seqs = sorted(set(rng.choice(dec, size=min(n_seq_sample, len(dec)), replace=False).tolist()) | set(chk))
    sub, sub_ten, tok = compact_layout(lay, ten, seqs)
    sub_cu = sub.cu_q_len
    want = []
    for i, s in enumerate(seqs):
        n = int(sub.q_len[i])
        if n == 1:
            want.append(int(sub_cu[i]))
        else:
            pick = rng.choice(n, size=min(n, n_chunk_tok), replace=False)
            pick = np.union1d(pick, [0, n - 1])
            want.extend((int(sub_cu[i]) + pick).tolist())
    _, _, ref = oracle_step(sub, sub_ten, tokens=want)
    got = out[torch.from_numpy(tok).cuda()]
    return compare(got, ref, tokens=want)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mistral_b512", "mistral_b512_window", "yi_b2048", "yi_b2048_o5043",
                                  "decode_only"])
def test_full_size_workloads(name):
    _full_size(name)


@pytest.mark.slow
@pytest.mark.parametrize("chunk,index", [(256, 31), (257, 0), (257, 31), (512, 7),
                                         (1024, 5), (2048, 3), (8192, 0)])
def test_chunk_sweep_batches(chunk, index):
    """The chunk-size sweep's batches: chunk `index` of an 8192-token prompt
    beside 32 decode rows at context 2048 (257 leaves a ragged last chunk of
    225 tokens and chunks that straddle pages)."""
    _full_size(None, seed=4, lay=workloads.chunk_sweep(chunk, index))


def test_wait_timeout_is_reported_and_context_survives():
    """A kernel wait that runs out ends the kernel with a status, not a hang:
    the library's bounded wait on a barrier nothing arrives at."""
    hb = lib()
    hb.hb_selftest_wait_timeout()
    with pytest.raises(hb.HbError) as e:
        hb.hb_check()
    assert e.value.status == 7
    hb.hb_check()                      # the word was cleared
    _full_check(workloads.tiny(0))     # the context still works


def test_flag_wait_timeout_is_reported_and_context_survives():
    """hb_step's append waits for its slot's flag with the same bounded wait:
    on a flag that is never raised it ends with a status, not a hang."""
    hb = lib()
    hb.hb_selftest_flag_timeout()
    with pytest.raises(hb.HbError) as e:
        hb.hb_check()
    assert e.value.status == 7
    hb.hb_check()
    _full_check(workloads.tiny(0))


def test_staged_step_through_host_buffers():
    """The packed host staging (one copy in, one out, on side streams) gives
    the same output as the device-resident step, and matches the oracle."""
    from chunked_prefill_decode_gb300.device import StepStaging
    hb = lib()
    lay = layout_from_rows(Shape(32, 8, 128), [(1, 700), (40, 300), (1, 33), (17, 17)], 21)
    ten = workloads.make_tensors(lay, 21)
    sh = lay.shape
    dev = torch.device("cuda:0")
    kc0, vc0, ref_out = gpu_step(lay, ten)
    kc, vc = ten.k_cache.to(dev).clone(), ten.v_cache.to(dev).clone()
    stg = StepStaging(lay.num_seqs, lay.total_q, lay.block_table.shape[1], lay.num_pages,
                      sh.num_q_heads, sh.num_kv_heads, sh.head_dim, device=dev)
    stg.h_q.copy_(ten.q)
    stg.h_k_new.copy_(ten.k_new)
    stg.h_v_new.copy_(ten.v_new)
    stg.h_cu_q_len.copy_(torch.from_numpy(lay.cu_q_len))
    stg.h_context_len.copy_(torch.from_numpy(lay.context_len))
    stg.h_block_table.copy_(torch.from_numpy(np.ascontiguousarray(lay.block_table)))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    stg.upload(s_in)
    main.wait_stream(s_in)
    plan, ws = hb.hb_plan(stg.batch, lay.q_len, lay.context_len, sms())
    hb.hb_kv_append(stg.batch, stg.k_new, stg.v_new, kc, vc)
    hb.hb_attention(stg.batch, plan, stg.q, kc, vc, 1.0 / math.sqrt(sh.head_dim), stg.out, ws)
    s_out.wait_stream(main)
    stg.download(s_out)
    s_out.synchronize()
    hb.hb_check()
    assert torch.equal(stg.h_out.view(torch.int16), ref_out.cpu().view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc0.view(torch.int16))
    _, _, ref = oracle_step(lay, ten)
    compare(stg.h_out, ref)


def test_hb_step_with_slots_in_flight():
    """hb_step: three slots, each with its own inputs (other q, k_new and
    v_new values over the same batch layout), stepped round-robin without
    the host waiting; after each slot's sync its output equals the
    device-resident append + attention on that slot's inputs, bit for bit,
    and matches the oracle."""
    from chunked_prefill_decode_gb300.device import StepStaging
    hb = lib()
    lay = layout_from_rows(Shape(32, 8, 128), [(1, 700), (40, 300), (1, 33), (17, 17), (1, 2000)], 22)
    sh = lay.shape
    dev = torch.device("cuda:0")
    base = workloads.make_tensors(lay, 22)
    kc, vc = base.k_cache.to(dev).clone(), base.v_cache.to(dev).clone()
    scale = 1.0 / math.sqrt(sh.head_dim)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    main = torch.cuda.current_stream(dev)
    ql = np.ascontiguousarray(lay.q_len, dtype=np.int32)
    cl = np.ascontiguousarray(lay.context_len, dtype=np.int32)
    slots, tens = [], []
    for k in range(3):
        ten = workloads.make_tensors(lay, 100 + k)
        ten = workloads.BatchTensors(ten.q, ten.k_new, ten.v_new, base.k_cache, base.v_cache)
        stg = StepStaging(lay.num_seqs, lay.total_q, lay.block_table.shape[1], lay.num_pages,
                          sh.num_q_heads, sh.num_kv_heads, sh.head_dim, device=dev)
        stg.h_q.copy_(ten.q)
        stg.h_k_new.copy_(ten.k_new)
        stg.h_v_new.copy_(ten.v_new)
        stg.h_cu_q_len.copy_(torch.from_numpy(lay.cu_q_len))
        stg.h_context_len.copy_(torch.from_numpy(lay.context_len))
        stg.h_block_table.copy_(torch.from_numpy(np.ascontiguousarray(lay.block_table)))
        stg.plan, stg.ws = hb.hb_plan(stg.batch, lay.q_len, lay.context_len, sms())
        stg.slot = hb.StepSlot()
        stg.bufs = stg.step_buffers(stg.plan, stg.ws)
        slots.append(stg)
        tens.append(ten)
    for i in range(9):
        stg = slots[i % 3]
        hb.hb_step(stg.batch, ql, cl, sms(), stg.slot, stg.bufs, kc, vc, scale, s_in, main, s_out)
    for k, stg in enumerate(slots):
        stg.slot.sync()
        _, _, ref_out = gpu_step(lay, tens[k])
        assert torch.equal(stg.h_out.view(torch.int16), ref_out.cpu().view(torch.int16))
        _, _, ref = oracle_step(lay, tens[k])
        compare(stg.h_out, ref)
    hb.hb_check()


def test_attention_right_after_the_kernel_that_writes_q():
    """hb_attention launched directly after an hb_linear that writes its q (no
    append in between) waits for that grid before it reads q; and directly
    after the append of another batch it also waits first."""
    from chunked_prefill_decode_gb300.device import device_batch
    hb = lib()
    lay = layout_from_rows(Shape(32, 8, 128), [(1, 3000)] * 6 + [(1, 700), (40, 300)], 25)
    ten = workloads.make_tensors(lay, 25)
    sh = lay.shape
    dev = torch.device("cuda:0")
    T = lay.total_q
    db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                      sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev)
    kc, vc = ten.k_cache.to(dev).clone(), ten.v_cache.to(dev).clone()
    hb.hb_kv_append(db.batch, ten.k_new.to(dev), ten.v_new.to(dev), kc, vc)
    plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms())
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(25)
    H = sh.num_q_heads * sh.head_dim
    x = torch.randn(T, 2048, generator=g).to(torch.bfloat16).to(dev)
    w = (torch.randn(H, 2048, generator=g) / math.sqrt(2048)).to(torch.bfloat16).to(dev)
    scale = 1.0 / math.sqrt(sh.head_dim)
    for _ in range(3):
        q = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        out = torch.full((T, sh.num_q_heads, sh.head_dim), float("nan"), dtype=torch.bfloat16,
                         device=dev)
        hb.hb_linear(x, w, [q])
        hb.hb_attention(db.batch, plan, q.view(T, sh.num_q_heads, sh.head_dim), kc, vc, scale,
                        out, ws)
        torch.cuda.synchronize()
        hb.hb_check()
        t2 = workloads.BatchTensors(q.view(T, sh.num_q_heads, sh.head_dim).cpu(), ten.k_new,
                                    ten.v_new, ten.k_cache, ten.v_cache)
        _, _, ref = oracle_step(lay, t2)
        compare(out, ref)
    # an append of another batch (a copy of the descriptors) right before:
    # the attention of this batch does not take it for its own
    db2 = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                       sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev)
    q = ten.q.to(dev)
    out = torch.full_like(q, float("nan"))
    hb.hb_kv_append(db2.batch, ten.k_new.to(dev), ten.v_new.to(dev), kc, vc)
    hb.hb_attention(db.batch, plan, q, kc, vc, scale, out, ws)
    torch.cuda.synchronize()
    hb.hb_check()
    _, _, ref = oracle_step(lay, ten)
    compare(out, ref)


def test_step_captured_in_a_cuda_graph():
    """Append + attention captured once in a CUDA graph (torch.cuda.graph) and
    replayed: the same output as the direct launches, replay after replay."""
    from chunked_prefill_decode_gb300.device import device_batch
    hb = lib()
    lay = layout_from_rows(Shape(32, 8, 128), [(1, 3000)] * 6 + [(1, 700), (40, 300)], 31)
    ten = workloads.make_tensors(lay, 31)
    sh = lay.shape
    dev = torch.device("cuda:0")
    db = device_batch(lay.q_len, lay.context_len, lay.block_table, lay.num_pages,
                      sh.num_q_heads, sh.num_kv_heads, sh.head_dim, sh.page_size, dev)
    q, kn, vn = (t.to(dev) for t in (ten.q, ten.k_new, ten.v_new))
    kc, vc = ten.k_cache.to(dev).clone(), ten.v_cache.to(dev).clone()
    plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms())
    scale = 1.0 / math.sqrt(sh.head_dim)
    out_direct = torch.full_like(q, float("nan"))
    hb.hb_kv_append(db.batch, kn, vn, kc, vc)
    hb.hb_attention(db.batch, plan, q, kc, vc, scale, out_direct, ws)
    torch.cuda.synchronize()
    hb.hb_check()
    out = torch.full_like(q, float("nan"))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        hb.hb_kv_append(db.batch, kn, vn, kc, vc)
        hb.hb_attention(db.batch, plan, q, kc, vc, scale, out, ws)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        hb.hb_check()
        assert torch.equal(out.view(torch.int16), out_direct.view(torch.int16))
    _, _, ref = oracle_step(lay, ten)
    compare(out, ref)


@pytest.mark.parametrize("seed", range(8))
def test_random_hybrid_batches(seed):
    """Seeded random hybrid batches (decode rows and chunks of any size, head
    geometries, windows): append bit-exact and attention within the bounds,
    every token checked against the oracle."""
    rng = np.random.default_rng(2000 + seed)
    geoms = [(8, 8, 64), (32, 8, 128), (56, 8, 128), (16, 2, 64), (64, 16, 128), (16, 1, 128),
             (32, 32, 128), (8, 1, 64)]
    hq, hkv, d = geoms[seed]
    rows = [(1, int(rng.integers(1, 2500))) for _ in range(int(rng.integers(0, 12)))]
    for _ in range(int(rng.integers(1, 3))):
        q = int(rng.integers(2, 400))
        rows.append((q, q + int(rng.integers(0, 1500))))
    rng.shuffle(rows)
    window = int(rng.choice([0, 0, 5, 300]))
    _full_check(layout_from_rows(Shape(hq, hkv, d, sliding_window=window),
                                 [tuple(r) for r in rows], 2000 + seed), seed=seed)
