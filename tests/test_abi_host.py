"""The C ABI on the host (no GPU): the library loads and exports every call
include/hb.h declares; argument errors come back as status codes; the plan
is checked against its own definition (coverage, splits, ordering)."""
import ctypes

import numpy as np
import pytest
import torch

from _hbutil import header_functions, host_batch, lib


def test_library_exports_every_declared_function():
    hb = lib()
    L = hb.load()
    declared = header_functions()
    assert "hb_kv_append" in declared and "hb_plan" in declared and "hb_attention" in declared
    for name in declared:
        assert hasattr(L, name), f"{name} declared in hb.h but not exported"
    assert set(hb.EXPORTED) == set(declared)


def test_status_strings():
    L = lib().load()
    for code, name in lib().STATUS_NAMES.items():
        assert L.hb_status_string(code).decode() == name


def test_timing_modes():
    L = lib().load()
    assert L.hb_timing_enable(3) == 1 and L.hb_timing_enable(-1) == 1   # HB_ERR_INVALID_ARG
    for mode in (1, 0, 2, 0):
        assert L.hb_timing_enable(mode) == 0
    ms = (ctypes.c_double * 3)()
    n = (ctypes.c_int32 * 3)()
    assert L.hb_timing_read(ms, n) == 0 and list(n) == [0, 0, 0]
    # per-launch durations: no records yet; bad kernel ids and NULLs refused
    cnt = ctypes.c_int32(-1)
    buf = (ctypes.c_float * 4)()
    assert L.hb_timing_durations(1, buf, 4, ctypes.byref(cnt)) == 0 and cnt.value == 0
    assert L.hb_timing_durations(3, buf, 4, ctypes.byref(cnt)) == 1
    assert L.hb_timing_durations(-1, buf, 4, ctypes.byref(cnt)) == 1
    assert L.hb_timing_durations(0, None, 4, ctypes.byref(cnt)) == 1
    assert L.hb_timing_durations(0, None, 0, ctypes.byref(cnt)) == 0


@pytest.mark.parametrize("field,value,status", [
    ("page_size", 8, 3), ("head_dim", 96, 3), ("num_kv_heads", 3, 2),
    ("num_q_heads", 0, 2), ("num_pages", 0, 2), ("max_pages_per_seq", 0, 2),
    ("num_seqs", -1, 2), ("total_q", -5, 2),
])
def test_bad_batch_is_rejected_on_the_host(field, value, status):
    hb = lib()
    b, ql, cl = host_batch(hb, [(1, 40), (5, 9)])
    setattr(b, field, value)
    with pytest.raises(hb.HbError) as e:
        hb.hb_plan_sizes(b, ql, cl, 148)
    assert e.value.status == status


def test_group_too_large_and_odd_kv_heads_unsupported():
    hb = lib()
    b, ql, cl = host_batch(hb, [(1, 40)], hq=34, hkv=2)
    with pytest.raises(hb.HbError) as e:
        hb.hb_plan_sizes(b, ql, cl, 148)
    assert e.value.status == 3
    b, ql, cl = host_batch(hb, [(1, 40)], hq=12, hkv=12)
    with pytest.raises(hb.HbError) as e:
        hb.hb_plan_sizes(b, ql, cl, 148)
    assert e.value.status == 3


@pytest.mark.parametrize("rows", [[(0, 5)], [(6, 5)], [(1, 4000)]])
def test_bad_rows_rejected(rows):
    hb = lib()
    b, ql, cl = host_batch(hb, rows, max_pages=8)
    with pytest.raises(hb.HbError) as e:
        hb.hb_plan_sizes(b, ql, cl, 148)
    assert e.value.status == 2


def test_total_q_mismatch_rejected():
    hb = lib()
    b, ql, cl = host_batch(hb, [(3, 9)])
    b.total_q = 4
    with pytest.raises(hb.HbError) as e:
        hb.hb_plan_sizes(b, ql, cl, 148)
    assert e.value.status == 2


def test_null_arguments():
    hb = lib()
    L = hb.load()
    assert L.hb_kv_append(None, None, None, None, None, None) == 1
    b, ql, cl = host_batch(hb, [(2, 9)])
    # total_q > 0 with NULL tensors
    assert L.hb_kv_append(ctypes.byref(b), None, None, None, None, None) == 1
    assert L.hb_attention(ctypes.byref(b), None, None, None, None, 1.0, None, None, None) == 1
    assert "NULL" in L.hb_last_error().decode()


def test_empty_batch_is_a_no_op():
    hb = lib()
    L = hb.load()
    b, ql, cl = host_batch(hb, [])
    assert L.hb_kv_append(ctypes.byref(b), None, None, None, None, None) == 0
    p, w = hb.hb_plan_sizes(b, ql, cl, 148)
    plan, _ = hb.hb_plan(b, ql, cl, 148, upload=False)
    assert hb.plan_header(plan)["num_decode_items"] == 0
    assert L.hb_attention(ctypes.byref(b), hb._ptr(plan), None, None, None, 1.0,
                          None, None, None) == 0


def test_attention_rejects_foreign_plan():
    hb = lib()
    L = hb.load()
    b, ql, cl = host_batch(hb, [(1, 50), (7, 7)])
    plan, _ = hb.hb_plan(b, ql, cl, 148, upload=False)
    b2, _, _ = host_batch(hb, [(1, 50), (8, 8)])
    assert L.hb_attention(ctypes.byref(b2), hb._ptr(plan), None, None, None, 1.0,
                          None, None, None) == 4
    junk = np.zeros_like(plan)
    assert L.hb_attention(ctypes.byref(b), hb._ptr(junk), None, None, None, 1.0,
                          None, None, None) == 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_cuda_calls_fail_cleanly_without_a_gpu():
    hb = lib()
    L = hb.load()
    b, ql, cl = host_batch(hb, [(2, 9)])
    buf = (ctypes.c_uint8 * 64)()
    ptr = ctypes.cast(buf, ctypes.c_void_p)
    aligned = ctypes.c_void_p((ptr.value + 15) // 16 * 16)
    st = L.hb_kv_append(ctypes.byref(b), aligned, aligned, aligned, aligned, None)
    assert st == 5


def _check_plan(rows, hq, hkv, d, sms, window=0):
    hb = lib()
    b, ql, cl = host_batch(hb, rows, hq=hq, hkv=hkv, d=d, window=window)
    plan, _ = hb.hb_plan(b, ql, cl, sms, upload=False)
    h = hb.plan_header(plan)
    dec, chk, offs = hb.plan_items(plan)
    g = hq // hkv
    kvhb = min(hkv, 8)
    assert h["decode_kvh_block"] == kvhb
    assert h["chunk_tokens_per_tile"] == 128 // g
    cu = np.concatenate([[0], np.cumsum(ql)])
    # decode: intervals are contiguous and together tile every decode row's
    # pages once per kv block; the CTAs' static ranges are equal (without a
    # dynamic tail the last may be shorter); the dynamic tail's intervals hold
    # at most as many pages as a static range, about 10 % of all pages
    grid, n_dyn = h["decode_grid"], h["num_decode_dynamic"]
    assert grid <= sms and offs[0] == 0 and offs[-1] == len(dec)
    assert len(offs) == (grid + n_dyn + 1 if grid else 1)
    assert (np.diff(offs) >= 1).all() if grid else len(dec) == 0
    pages = [int(sum(dec[i, 3] - dec[i, 2] for i in range(offs[c], offs[c + 1])))
             for c in range(grid + n_dyn)]
    if grid:
        st = pages[:grid]
        if n_dyn:
            assert all(x == st[0] for x in st)
            assert max(pages[grid:]) <= max(4, st[0]) and 4 <= max(pages[grid:])
            assert sum(pages[grid:]) <= 0.1 * sum(pages) + grid
        else:
            assert all(x == st[0] for x in st[:-1]) and st[-1] <= st[0]
    cover = {}
    for seq, kvh0, pb, pe, split, ns, slot, mid, ctx, tok, _, _ in dec:
        assert ql[seq] == 1 and 0 <= pb < pe and kvh0 % kvhb == 0
        assert ctx == cl[seq] and tok == cu[seq]
        cover.setdefault((seq, kvh0), []).append((pb, pe, split, ns, slot, mid))
    slots = set()
    for s in range(len(rows)):
        if ql[s] != 1:
            continue
        npg = -(-cl[s] // 16)
        first = (cl[s] - window) // 16 if 0 < window < cl[s] else 0
        for kvh0 in range(0, hkv, kvhb):
            parts = sorted(cover[(s, kvh0)])
            assert parts[0][0] == first and parts[-1][1] == npg
            assert all(a[1] == b_[0] for a, b_ in zip(parts, parts[1:]))
            ns = parts[0][3]
            assert len(parts) == ns and [p[2] for p in parts] == list(range(ns))
            assert len({(p[4], p[5]) for p in parts}) == 1
            if ns > 1:
                assert parts[0][4] not in slots
                slots.add(parts[0][4])
    # chunk items cover every (token, kv head) of every chunk row once; an
    # item holds two query tiles when there are enough tiles to fill the SMs
    # twice, and otherwise whichever of pairs and single tiles the plan
    # estimates to end first
    tpt = 128 // g
    n_tiles = sum(-(-int(q) // tpt) * hkv for q in ql if q > 1)
    tpi = 2 if n_tiles >= 2 * sms or any(int(c[3]) > tpt for c in chk) else 1
    seen = set()
    groups = {}
    for seq, kvh, t0, nt, end, q0, qn, ctx, kb, split, ns, slot, mid, *_ in chk:
        assert ql[seq] > 1 and 1 <= nt <= tpi * tpt and t0 % (tpi * tpt) == 0
        assert q0 == cu[seq] and qn == ql[seq] and ctx == cl[seq]
        assert 1 <= ns <= 16 and 0 <= split < ns and 0 <= kb < end
        if ns > 1:
            assert end - kb >= 4                   # no piece below 4 key tiles
        groups.setdefault((seq, kvh, t0), []).append((split, kb, end, ns, slot, mid, nt))
    slots, merges = set(), set()
    for (seq, kvh, t0), parts in groups.items():
        parts.sort()
        ns = parts[0][3]
        nt = parts[0][6]
        off = cl[seq] - ql[seq]
        # the pieces tile the key range of the query tile(s) exactly once
        assert [p[0] for p in parts] == list(range(ns))
        kb0 = max(0, off + t0 - window + 1) // 128 if window > 0 else 0
        assert parts[0][1] == kb0 and parts[-1][2] == -(-(off + t0 + nt) // 128)
        assert all(a[2] == b_[1] for a, b_ in zip(parts, parts[1:]))
        assert len({(p[3], p[4], p[5], p[6]) for p in parts}) == 1
        if ns > 1:
            assert parts[0][5] not in merges
            merges.add(parts[0][5])
            # one partial state per piece and query tile (a pair has two)
            tiles = 2 if nt > tpt else 1
            rng_ = set(range(parts[0][4], parts[0][4] + ns * tiles))
            assert not (rng_ & slots)
            slots |= rng_
        for t in range(t0, t0 + nt):
            assert (seq, kvh, t) not in seen
            seen.add((seq, kvh, t))
    assert len(seen) == sum(int(q) * hkv for q in ql if q > 1)
    assert h["num_chunk_slots"] == len(slots) and h["num_chunk_merges"] == len(merges)
    assert slots == set(range(len(slots))) and merges == set(range(len(merges)))
    lengths = [c[4] - c[8] for c in chk]
    assert lengths == sorted(lengths, reverse=True)
    # the launch takes a pairs-only kernel when every chunk item is an unsplit
    # pair of query tiles (bit 0), and one that writes softmax weights in two
    # terms when some item's first row sees at most 256 keys (bit 1)
    def first_keys(c):
        k = int(c[7]) - int(c[6]) + int(c[2]) + 1
        return min(window, k) if window > 0 else k
    pairs_only = len(chk) > 0 and all(int(c[3]) > tpt and int(c[10]) == 1 for c in chk)
    few = any(first_keys(c) <= 256 for c in chk)
    assert h["chunk_pairs_only"] == (1 if pairs_only else 0) | (2 if few else 0)
    return h


@pytest.mark.parametrize("name", ["tiny", "mistral_b512", "mistral_b512_window", "yi_b2048", "yi_b2048_o5043",
                                  "decode_only"])
def test_plan_covers_workloads(name):
    from chunked_prefill_decode_gb300 import workloads
    lay = workloads.WORKLOADS[name]()
    sh = lay.shape
    rows = list(zip(lay.q_len.tolist(), lay.context_len.tolist()))
    h = _check_plan(rows, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, 152,
                    window=sh.sliding_window)


def test_plan_of_a_decode_batch_after_a_chunk_batch():
    """The plan's working arrays are reused from call to call on a thread: a
    batch without chunk rows planned after one with many has no chunk item."""
    from chunked_prefill_decode_gb300 import workloads
    for name in ("yi_b2048", "decode_only", "mistral_b512", "decode_only"):
        lay = workloads.WORKLOADS[name]()
        sh = lay.shape
        rows = list(zip(lay.q_len.tolist(), lay.context_len.tolist()))
        h = _check_plan(rows, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, 152)
        if name == "decode_only":
            assert h["num_chunk_items"] == 0


def test_plan_edge_shapes():
    _check_plan([(1, 1), (1, 16), (1, 17), (2, 2), (17, 17), (129, 300)], 8, 8, 64, 4)
    _check_plan([(1, 5000), (257, 8192)], 56, 8, 128, 152)
    _check_plan([(1, 333), (9, 40)], 16, 16, 128, 8)    # 2 kv blocks of 8
    _check_plan([(1, 100), (3, 3)], 4, 2, 64, 152)      # kv block of 2


@pytest.mark.parametrize("window", [1, 15, 16, 17, 300, 4096, 100000])
def test_plan_with_sliding_window(window):
    """Decode ranges start at the window's first page; chunk items start at
    the first key tile their first row sees; the header records the window."""
    rows = [(1, 1), (1, 17), (1, 5000), (1, 333), (257, 8192), (40, 45), (1, 3000)]
    h = _check_plan(rows, 32, 8, 128, 148, window=window)
    assert h["sliding_window"] == window
    _check_plan(rows, 8, 8, 64, 8, window=window)


def test_attention_rejects_plan_of_another_window():
    hb = lib()
    L = hb.load()
    b, ql, cl = host_batch(hb, [(1, 500), (9, 90)], window=64)
    plan, _ = hb.hb_plan(b, ql, cl, 148, upload=False)
    b2, _, _ = host_batch(hb, [(1, 500), (9, 90)], window=0)
    assert L.hb_attention(ctypes.byref(b2), hb._ptr(plan), None, None, None, 1.0,
                          None, None, None) == 4


def test_negative_window_and_reserved_field_are_rejected():
    hb = lib()
    L = hb.load()
    b, ql, cl = host_batch(hb, [(1, 50)])
    b.sliding_window = -1
    assert L.hb_plan(ctypes.byref(b), hb._ptr(ql), hb._ptr(cl), 148, None,
                     ctypes.byref(ctypes.c_size_t(0)), None,
                     ctypes.byref(ctypes.c_size_t(0)), None) == 2
    b.sliding_window, b.reserved = 0, 7
    assert L.hb_plan(ctypes.byref(b), hb._ptr(ql), hb._ptr(cl), 148, None,
                     ctypes.byref(ctypes.c_size_t(0)), None,
                     ctypes.byref(ctypes.c_size_t(0)), None) == 1


def test_plan_splits_short_chunks_at_long_offsets():
    """A 256-token chunk at offset 7936 (64 query tiles of 64 key tiles) cannot
    fill 148 SMs as whole tiles: its key ranges are split; a chunk with enough
    tiles to pair is not."""
    h = _check_plan([(256, 8192)], 32, 8, 128, 148)
    assert h["num_chunk_merges"] > 0 and h["num_chunk_slots"] >= 2 * h["num_chunk_merges"]
    h = _check_plan([(1, 2048)] * 32 + [(256, 8192)], 32, 8, 128, 148)
    assert h["num_chunk_merges"] > 0
    h = _check_plan([(4096, 8192)], 32, 8, 128, 148)
    assert h["num_chunk_merges"] == 0
    # short key ranges are never split below 4 tiles per piece
    h = _check_plan([(64, 64 + 200)], 8, 8, 64, 148)
    assert h["num_chunk_merges"] == 0


def test_linear_argument_checks():
    """hb_linear's host-side checks (no GPU needed: they come first)."""
    hb = lib()
    L = hb.load()
    buf = (ctypes.c_uint8 * 256)()
    base = ctypes.cast(buf, ctypes.c_void_p).value
    a16 = ctypes.c_void_p((base + 15) // 16 * 16)
    odd = ctypes.c_void_p(a16.value + 2)

    def call(x, w, M, N, K, epi, cols, ys=None):
        o = hb.HbLinearOut()
        for i in range(3):
            o.cols[i] = cols[i]
            o.y[i] = (ys[i] if ys else a16).value if cols[i] else None
        return L.hb_linear(x, w, M, N, K, epi, ctypes.byref(o), None, 0, None)

    assert L.hb_linear(a16, a16, 4, 256, 64, 0, None, None, 0, None) == 1  # out NULL
    assert call(a16, a16, 4, 256, 64, 3, (256, 0, 0)) == 1                # unknown epilogue
    assert call(a16, a16, 4, 256, 96, 0, (256, 0, 0)) == 2                # K % 64
    assert call(a16, a16, 4, 320, 64, 0, (320, 0, 0)) == 2                # N % 256
    assert call(a16, a16, 4, 512, 64, 0, (256, 0, 0)) == 2                # cols sum != N
    assert call(a16, a16, 4, 512, 64, 0, (256, 128, 128)) == 2            # cols % 256
    assert call(a16, a16, 4, 512, 64, 1, (512, 0, 0)) == 2                # gated: cols = F
    assert call(odd, a16, 4, 256, 64, 0, (256, 0, 0)) == 1                # misaligned x
    assert call(a16, a16, 4, 256, 64, 0, (256, 0, 0), ys=[odd, a16, a16]) == 1
    assert call(a16, a16, -1, 256, 64, 0, (256, 0, 0)) == 2               # M < 0
    assert call(a16, a16, 0, 768, 64, 0, (256, 512, 0)) == 0              # M = 0: nothing to do
    assert call(a16, a16, 0, 512, 64, 1, (256, 0, 0)) == 0


def test_linear_workspace_size():
    """Split-K only when the 256 x 256 tiles (one per pair of CTAs) cannot
    fill half the 76 pairs of 152 SMs: then up to 16 pieces of at least four
    K blocks, about one piece per pair; the workspace holds a fixed 4 KB
    counter region, then one fp32 half tile (128 rows x 256 columns) per
    (tile, CTA of the pair, piece)."""
    hb = lib()
    L = hb.load()
    half = 128 * 256 * 4
    # 2 x 16 tiles on 76 pairs: 2 pieces of 32 K blocks
    assert L.hb_linear_workspace_size(512, 4096, 4096, 0, 152) == 4096 + 2 * 32 * 2 * half
    assert L.hb_linear_workspace_size(512, 4096, 14336, 0, 152) == 4096 + 2 * 32 * 2 * half
    # one tile, 64 K blocks: 16 pieces
    assert L.hb_linear_workspace_size(1, 256, 4096, 0, 152) == 4096 + 16 * 1 * 2 * half
    # enough tiles (2 x 24 = 48 > 76 / 2), or too little K to split: none
    assert L.hb_linear_workspace_size(512, 6144, 4096, 0, 152) == 0
    assert L.hb_linear_workspace_size(8192, 4096, 4096, 0, 152) == 0
    assert L.hb_linear_workspace_size(256, 28672, 4096, 1, 152) == 0
    assert L.hb_linear_workspace_size(1, 256, 256, 0, 152) == 0
    # gated: tiles of 128 output columns from [gate; up]; 2 x 2 tiles, 16 K
    # blocks: 4 pieces of 4
    assert L.hb_linear_workspace_size(300, 512, 1024, 1, 152) == 4096 + 4 * 4 * 2 * half
    # invalid shapes: 0
    assert L.hb_linear_workspace_size(4, 300, 64, 0, 152) == 0
    assert L.hb_linear_workspace_size(4, 256, 100, 0, 152) == 0


@pytest.mark.parametrize("seed", range(32))
def test_plan_invariants_on_random_batches(seed):
    """Seeded random hybrid batches (mixes of decode rows and chunks of every
    size, several head geometries, SM counts and windows): every plan tiles
    each decode row's pages and each chunk's (token, kv head) pairs exactly
    once, with consistent split-KV pieces (the same checks as above)."""
    rng = np.random.default_rng(1000 + seed)
    geoms = [(8, 8, 64), (32, 8, 128), (56, 8, 128), (16, 2, 64), (64, 16, 128), (16, 1, 128)]
    hq, hkv, d = geoms[seed % len(geoms)]
    n_dec = int(rng.integers(0, 40))
    n_chk = int(rng.integers(0 if n_dec else 1, 4))
    rows = [(1, int(rng.integers(1, 9000))) for _ in range(n_dec)]
    for _ in range(n_chk):
        q = int(rng.integers(2, 3000))
        rows.append((q, q + int(rng.integers(0, 6000))))
    rng.shuffle(rows)
    sms = int(rng.choice([1, 7, 64, 148, 152]))
    window = int(rng.choice([0, 0, 0, 1, 37, 1024]))
    _check_plan([tuple(r) for r in rows], hq, hkv, d, sms, window=window)


@pytest.mark.parametrize("rows,geom", [([(1, 40), (64, 500), (1, 3000)], (32, 8, 128)),
                                       ([(7, 7)], (8, 8, 64)), ([(1, 1)] * 33, (56, 8, 128))])
def test_step_layout_matches_the_staging_buffers(rows, geom):
    """hb_step's packed input block has the layout the Python staging
    buffers fill: q, k_new, v_new, cu_q_len, context_len, block_table, each
    on a 256-byte boundary."""
    from chunked_prefill_decode_gb300.device import StepStaging
    hb = lib()
    hq, hkv, d = geom
    b, ql, cl = host_batch(hb, rows, hq=hq, hkv=hkv, d=d)
    offs, total = hb.hb_step_layout(b)
    parts, want = StepStaging.layout(b.num_seqs, b.total_q, b.max_pages_per_seq, hq, hkv, d)
    assert offs == [p[3] for p in parts] and total == want
    assert all(o % 256 == 0 for o in offs)


def test_step_argument_errors_need_no_gpu():
    hb = lib()
    L = hb.load()
    b, ql, cl = host_batch(hb, [(1, 40)])
    bufs = hb.HbStepBuffers()
    assert L.hb_step(ctypes.byref(b), hb._ptr(ql), hb._ptr(cl), 148, None, ctypes.byref(bufs),
                     None, None, 1.0, None, None, None) == 1       # NULL slot
    assert L.hb_step_slot_sync(None) == 1
    L.hb_step_slot_destroy(None)                                   # a no-op
    offs = (ctypes.c_size_t * 6)()
    n = ctypes.c_size_t(0)
    b.num_q_heads = 0
    assert L.hb_step_layout(ctypes.byref(b), offs, ctypes.byref(n)) == 2
    assert L.hb_step_layout(None, offs, ctypes.byref(n)) == 1
