"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties oracle.paged_attention to something the pages or mathematics
fix: a pure-Python brute force, closed forms, chunked == unchunked prefill
(chunking changes cost, not the result), decode row == last prefill row,
causality, page-permutation invariance, GQA == expanded multi-head attention,
the split-softmax merge identity and torch's fp64 scaled_dot_product_attention.
The mutation tests at the end plant plausible mistakes in the oracle and
check that a pin catches each one.
"""
import math

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from oracle.brute import attention_bruteforce

P = 4  # small page size keeps page-boundary crossings frequent in tiny cases


def _pools(rng, num_pages, hkv, d, page=P):
    k = rng.standard_normal((num_pages, page, hkv, d))
    v = rng.standard_normal((num_pages, page, hkv, d))
    return k, v


def _random_batch(rng, rows, hq, hkv, d, page=P, extra_pages=3):
    """rows = [(q_len, ctx)]; random scattered pages; float64 values."""
    pages_per = [-(-c // page) for _, c in rows]
    num_pages = sum(pages_per) + extra_pages
    perm = rng.permutation(num_pages)
    bt = np.full((len(rows), max(pages_per)), -1, dtype=np.int64)
    k = 0
    for s, n in enumerate(pages_per):
        bt[s, :n] = perm[k:k + n]
        k += n
    kp, vp = _pools(rng, num_pages, hkv, d, page)
    T = sum(q for q, _ in rows)
    q = rng.standard_normal((T, hq, d))
    ql = np.array([r[0] for r in rows])
    cl = np.array([r[1] for r in rows])
    return q, kp, vp, ql, cl, bt


def _attn(q, kp, vp, ql, cl, bt, hq, hkv, scale, page=P, **kw):
    return pa.attention(q, kp, vp, ql, cl, bt, page, hq, hkv, scale, **kw)


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_numpy_oracle_matches_bruteforce(seed):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 4, 2, 8
    rows = [(1, int(rng.integers(1, 13))),
            (int(rng.integers(2, 9)), int(rng.integers(9, 21))),
            (int(rng.integers(1, 6)), 5)]
    rows = [(min(a, b), b) for a, b in rows]
    q, kp, vp, ql, cl, bt = _random_batch(rng, rows, hq, hkv, d)
    scale = 1 / math.sqrt(d)
    ref = np.array(attention_bruteforce(q, kp, vp, ql, cl, bt, P, hq, hkv, scale))
    out = _attn(q, kp, vp, ql, cl, bt, hq, hkv, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_chunked_prefill_equals_unchunked():
    """Prefilling a prompt in N chunks gives the unchunked result, for chunk
    sizes that straddle page boundaries."""
    rng = np.random.default_rng(11)
    hq, hkv, d, L = 4, 2, 8, 37
    num_pages = -(-L // P) + 2
    bt = rng.permutation(num_pages)[None, : -(-L // P)]
    q = rng.standard_normal((L, hq, d))
    kn = rng.standard_normal((L, hkv, d))
    vn = rng.standard_normal((L, hkv, d))
    empty = np.full((num_pages, P, hkv, d), np.nan)
    scale = 0.3
    kf, vf = pa.kv_append(empty, empty, kn, vn, [L], [L], bt, P)
    full = _attn(q, kf, vf, [L], [L], bt, hq, hkv, scale)
    for c in (1, 3, 4, 5, 16, 17, L):
        kp, vp = empty.copy(), empty.copy()
        outs = []
        for start in range(0, L, c):
            n = min(c, L - start)
            sl = slice(start, start + n)
            kp, vp = pa.kv_append(kp, vp, kn[sl], vn[sl], [n], [start + n], bt, P)
            outs.append(_attn(q[sl], kp, vp, [n], [start + n], bt, hq, hkv, scale))
        np.testing.assert_allclose(np.concatenate(outs), full, rtol=0, atol=1e-13)
        np.testing.assert_array_equal(np.isnan(kp), np.isnan(kf))
        np.testing.assert_array_equal(np.nan_to_num(kp), np.nan_to_num(kf))


def test_decode_row_equals_last_prefill_row():
    rng = np.random.default_rng(12)
    hq, hkv, d, L = 6, 3, 8, 23
    num_pages = -(-L // P) + 1
    bt = rng.permutation(num_pages)[None, : -(-L // P)]
    q = rng.standard_normal((L, hq, d))
    kn = rng.standard_normal((L, hkv, d))
    vn = rng.standard_normal((L, hkv, d))
    empty = np.zeros((num_pages, P, hkv, d))
    kf, vf = pa.kv_append(empty, empty, kn, vn, [L], [L], bt, P)
    full = _attn(q, kf, vf, [L], [L], bt, hq, hkv, 0.5)
    kp, vp = pa.kv_append(empty, empty, kn[:-1], vn[:-1], [L - 1], [L - 1], bt, P)
    kp, vp = pa.kv_append(kp, vp, kn[-1:], vn[-1:], [1], [L], bt, P)
    dec = _attn(q[-1:], kp, vp, [1], [L], bt, hq, hkv, 0.5)
    np.testing.assert_allclose(dec[0], full[-1], rtol=0, atol=1e-14)


def test_causality_past_outputs_ignore_future_tokens():
    rng = np.random.default_rng(13)
    hq, hkv, d, L, p = 4, 4, 8, 20, 9
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(L, L)], hq, hkv, d)
    base = _attn(q, kp, vp, ql, cl, bt, hq, hkv, 0.4)
    q2, k2, v2 = q.copy(), kp.copy(), vp.copy()
    q2[p + 1:] += 5.0
    for t in range(p + 1, L):
        k2[bt[0, t // P], t % P] = rng.standard_normal((hkv, d)) * 7
        v2[bt[0, t // P], t % P] = rng.standard_normal((hkv, d)) * 7
    pert = _attn(q2, k2, v2, ql, cl, bt, hq, hkv, 0.4)
    np.testing.assert_array_equal(pert[: p + 1], base[: p + 1])
    assert not np.allclose(pert[p + 1:], base[p + 1:])


def test_constant_v_returns_v():
    rng = np.random.default_rng(14)
    hq, hkv, d = 4, 2, 8
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(1, 29), (7, 13)], hq, hkv, d)
    c = rng.standard_normal((hkv, d))
    vp[:] = c
    out = _attn(q, kp, vp, ql, cl, bt, hq, hkv, 1.7)
    expect = np.repeat(c, hq // hkv, axis=0)
    for t in range(out.shape[0]):
        np.testing.assert_allclose(out[t], expect, rtol=1e-14, atol=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(15)
    hq, hkv, d = 2, 1, 8
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(5, 11)], hq, hkv, d)
    q[:] = 0
    out = _attn(q, kp, vp, ql, cl, bt, hq, hkv, 1.0)
    V = pa.gather_logical(vp, bt[0], 11, P)[:, 0]
    for j in range(5):
        p = 11 - 5 + j
        np.testing.assert_allclose(out[j, 0], V[: p + 1].mean(axis=0), atol=1e-14)


def test_single_key_gives_that_value():
    rng = np.random.default_rng(16)
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(1, 1)], 3, 3, 8)
    out = _attn(q, kp, vp, ql, cl, bt, 3, 3, 0.9)
    np.testing.assert_array_equal(out[0], vp[bt[0, 0], 0])


def test_two_keys_closed_form():
    """o = (v0 + e^(s1 - s0) v1) / (1 + e^(s1 - s0))."""
    rng = np.random.default_rng(17)
    d = 8
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(1, 2)], 1, 1, d)
    scale = 0.25
    k0, k1 = kp[bt[0, 0], 0, 0], kp[bt[0, 0], 1, 0]
    v0, v1 = vp[bt[0, 0], 0, 0], vp[bt[0, 0], 1, 0]
    delta = scale * (q[0, 0] @ k1 - q[0, 0] @ k0)
    e = math.exp(delta)
    expect = (v0 + e * v1) / (1 + e)
    out = _attn(q, kp, vp, ql, cl, bt, 1, 1, scale)
    np.testing.assert_allclose(out[0, 0], expect, rtol=1e-13, atol=1e-14)


def test_physical_page_permutation_invariance():
    rng = np.random.default_rng(18)
    hq, hkv, d = 4, 2, 8
    rows = [(1, 17), (6, 6), (3, 14)]
    q, kp, vp, ql, cl, bt = _random_batch(rng, rows, hq, hkv, d, extra_pages=0)
    out = _attn(q, kp, vp, ql, cl, bt, hq, hkv, 0.3)
    # move every page to a new physical index; the block table follows
    perm = rng.permutation(kp.shape[0])
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1)
    out2 = _attn(q, kp2, vp2, ql, cl, bt2, hq, hkv, 0.3)
    np.testing.assert_array_equal(out, out2)


def test_gqa_equals_expanded_multihead():
    """GQA with contiguous groups (kv head = h // g) equals multi-head
    attention whose kv heads are those kv heads repeated g times each."""
    rng = np.random.default_rng(19)
    hq, hkv, d = 6, 2, 8
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(1, 9), (4, 10)], hq, hkv, d)
    g = hq // hkv
    kx, vx = np.repeat(kp, g, axis=2), np.repeat(vp, g, axis=2)
    a = _attn(q, kp, vp, ql, cl, bt, hq, hkv, 0.35)
    b = _attn(q, kx, vx, ql, cl, bt, hq, hq, 0.35)
    np.testing.assert_array_equal(a, b)


def test_split_softmax_merge_identity():
    rng = np.random.default_rng(20)
    s = rng.standard_normal(50) * 3
    v = rng.standard_normal((50, 8))
    w = np.exp(s - s.max())
    full = (w / w.sum()) @ v
    cuts = [0, 7, 16, 33, 50]
    states = [pa.partial_softmax_state(s[a:b], v[a:b]) for a, b in zip(cuts, cuts[1:])]
    np.testing.assert_allclose(pa.merge_partial_states(states), full, atol=1e-14)


def test_matches_torch_sdpa_with_bottom_right_mask():
    """Contiguous single sequence (identity block table) against torch's fp64
    scaled_dot_product_attention with an explicit bottom-right causal mask."""
    rng = np.random.default_rng(21)
    hq, hkv, d, ctx, ql = 4, 4, 16, 30, 11
    num_pages = -(-ctx // P)
    bt = np.arange(num_pages)[None]
    kp, vp = _pools(rng, num_pages, hkv, d)
    q = rng.standard_normal((ql, hq, d))
    scale = 1 / math.sqrt(d)
    out = _attn(q, kp, vp, [ql], [ctx], bt, hq, hkv, scale)
    K = torch.from_numpy(kp.reshape(-1, hkv, d)[:ctx]).permute(1, 0, 2)
    V = torch.from_numpy(vp.reshape(-1, hkv, d)[:ctx]).permute(1, 0, 2)
    Q = torch.from_numpy(q).permute(1, 0, 2)
    pos = torch.arange(ctx - ql, ctx)[:, None]
    mask = torch.arange(ctx)[None, :] <= pos
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q, K, V, attn_mask=mask, scale=scale).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_append_scatter_then_gather_and_sentinels():
    rng = np.random.default_rng(22)
    hkv, d = 2, 4
    rows = [(3, 9), (1, 5), (5, 5)]
    num_pages = 10
    perm = rng.permutation(num_pages)
    bt = np.array([perm[0:3], [perm[3], perm[4], -1], [perm[5], perm[6], -1]])
    sentinel = np.uint16(0x7FC1)
    pool = np.full((num_pages, P, hkv, d), sentinel, dtype=np.uint16)
    T = sum(r[0] for r in rows)
    kn = rng.integers(0, 2 ** 16, size=(T, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 2 ** 16, size=(T, hkv, d), dtype=np.uint16)
    ql = [r[0] for r in rows]
    cl = [r[1] for r in rows]
    kp, vp = pa.kv_append(pool, pool, kn, vn, ql, cl, bt, P)
    written = np.zeros((num_pages, P), dtype=bool)
    start = 0
    for s, (q, c) in enumerate(rows):
        got = pa.gather_logical(kp, bt[s], c, P)[c - q:]
        np.testing.assert_array_equal(got, kn[start:start + q])
        got = pa.gather_logical(vp, bt[s], c, P)[c - q:]
        np.testing.assert_array_equal(got, vn[start:start + q])
        for t in range(c - q, c):
            written[bt[s, t // P], t % P] = True
        start += q
    assert (kp[~written] == sentinel).all() and (vp[~written] == sentinel).all()


def test_bf16_decode_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F80, 0x0001], dtype=np.uint16)
    vals = pa.bf16_to_f64(bits)
    assert vals[0] == 1.0 and vals[1] == -1.0 and vals[2] == 0.0
    assert vals[3] == 3.140625 and math.isinf(vals[4])
    assert vals[5] == 2.0 ** -133
    t = torch.tensor([1.5, -2.25, 3.1], dtype=torch.bfloat16)
    np.testing.assert_array_equal(
        pa.bf16_to_f64(t.view(torch.int16).numpy().view(np.uint16)),
        t.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# Planted mistakes: each must be caught by at least one pin above.
# ---------------------------------------------------------------------------

def test_pin_catches_top_left_causal_alignment(monkeypatch):
    """The classic slip: aligning the causal mask to the first key instead of
    to the absolute position of each new token."""
    monkeypatch.setattr(pa, "query_positions",
                        lambda q, c: np.arange(q, dtype=np.int64))
    with pytest.raises(AssertionError):
        test_chunked_prefill_equals_unchunked()
    with pytest.raises(AssertionError):
        test_matches_torch_sdpa_with_bottom_right_mask()
    with pytest.raises(AssertionError):
        test_decode_row_equals_last_prefill_row()


def test_pin_catches_off_by_one_append(monkeypatch):
    real = pa.new_token_positions
    monkeypatch.setattr(pa, "new_token_positions", lambda q, c: real(q, c) + 1)
    with pytest.raises((AssertionError, IndexError)):
        test_append_scatter_then_gather_and_sentinels()


def test_pin_catches_interleaved_gqa_mapping(monkeypatch):
    rng = np.random.default_rng(23)
    hq, hkv, d = 4, 2, 8
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(2, 7)], hq, hkv, d)
    ref = np.array(attention_bruteforce(q, kp, vp, ql, cl, bt, P, hq, hkv, 0.5))
    # a wrong oracle that maps q head h to kv head h % Hkv
    perm = [0, 2, 1, 3]
    wrong = _attn(q[:, perm], kp, vp, ql, cl, bt, hq, hkv, 0.5)[:, perm]
    assert not np.allclose(wrong, ref)


def test_pin_catches_dropped_scale(monkeypatch):
    rng = np.random.default_rng(24)
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(3, 9)], 2, 1, 8)
    ref = np.array(attention_bruteforce(q, kp, vp, ql, cl, bt, P, 2, 1, 0.2))
    wrong = _attn(q, kp, vp, ql, cl, bt, 2, 1, 1.0)
    assert not np.allclose(wrong, ref, atol=1e-6)


def test_pin_catches_transposed_page_index(monkeypatch):
    """Swapping page and slot roles in the gather breaks the brute-force pin."""
    rng = np.random.default_rng(25)
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(2, 10)], 2, 2, 8)
    ref = np.array(attention_bruteforce(q, kp, vp, ql, cl, bt, P, 2, 2, 0.5))

    def wrong_gather(pool, row, n, page, start=0):
        pos = np.arange(start, n)
        return np.asarray(pool)[np.asarray(row)[pos % len(row)], pos // len(row) % page]
    monkeypatch.setattr(pa, "gather_logical", wrong_gather)
    out = _attn(q, kp, vp, ql, cl, bt, 2, 2, 0.5)
    assert not np.allclose(out, ref)


def test_pin_catches_merge_without_rescale(monkeypatch):
    """A merge that adds the pieces' sums without bringing them to the common
    maximum (exp(m_i - m)) breaks the split-softmax identity."""
    def wrong_merge(states):
        return sum(st[2] for st in states) / sum(st[1] for st in states)
    monkeypatch.setattr(pa, "merge_partial_states", wrong_merge)
    with pytest.raises(AssertionError):
        test_split_softmax_merge_identity()


def test_pin_catches_merge_that_drops_a_piece(monkeypatch):
    real = pa.merge_partial_states
    monkeypatch.setattr(pa, "merge_partial_states", lambda states: real(states[:-1]))
    with pytest.raises(AssertionError):
        test_split_softmax_merge_identity()


# --------------------------------------------------------------- sliding window
@pytest.mark.parametrize("seed,window", [(0, 1), (1, 3), (2, 5), (3, 9)])
def test_windowed_oracle_matches_bruteforce(seed, window):
    rng = np.random.default_rng(100 + seed)
    hq, hkv, d = 4, 2, 8
    rows = [(1, 11), (6, 17), (3, 3), (1, 2)]
    q, kp, vp, ql, cl, bt = _random_batch(rng, rows, hq, hkv, d)
    ref = np.array(attention_bruteforce(q, kp, vp, ql, cl, bt, P, hq, hkv, 0.3, window=window))
    out = _attn(q, kp, vp, ql, cl, bt, hq, hkv, 0.3, window=window)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_window_covering_the_context_is_full_attention():
    rng = np.random.default_rng(110)
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(1, 9), (5, 14)], 2, 2, 8)
    full = _attn(q, kp, vp, ql, cl, bt, 2, 2, 0.4)
    for w in (14, 15, 1000):
        np.testing.assert_array_equal(_attn(q, kp, vp, ql, cl, bt, 2, 2, 0.4, window=w), full)


def test_window_of_one_returns_own_value():
    """Closed form: with W = 1 each query sees only its own key, so o = v_p."""
    rng = np.random.default_rng(111)
    rows = [(1, 9), (5, 14)]
    q, kp, vp, ql, cl, bt = _random_batch(rng, rows, 4, 2, 8)
    out = _attn(q, kp, vp, ql, cl, bt, 4, 2, 0.4, window=1)
    r = 0
    for s, (qn, c) in enumerate(rows):
        for j in range(qn):
            p = c - qn + j
            v = vp[bt[s, p // P], p % P]          # [Hkv, D]
            np.testing.assert_allclose(out[r], np.repeat(v, 2, axis=0), rtol=0, atol=1e-15)
            r += 1


def test_windowed_chunked_prefill_equals_unchunked():
    """Chunking changes cost, not the result -- with a window as well."""
    rng = np.random.default_rng(112)
    L, W, hq, hkv, d = 23, 6, 2, 1, 8
    kp, vp = _pools(rng, 8, hkv, d)
    bt = np.array([rng.permutation(8)[:6]])
    qs = rng.standard_normal((L, hq, d))
    full = _attn(qs, kp, vp, [L], [L], bt, hq, hkv, 0.5, window=W)
    for c in (1, 4, 5, 9):
        got = []
        for o in range(0, L, c):
            n = min(c, L - o)
            got.append(_attn(qs[o:o + n], kp, vp, [n], [o + n], bt, hq, hkv, 0.5, window=W))
        np.testing.assert_allclose(np.concatenate(got), full, rtol=0, atol=1e-12)


def test_windowed_matches_torch_sdpa_band_mask():
    """One contiguous sequence: torch fp64 SDPA with an explicit band mask."""
    rng = np.random.default_rng(113)
    ctx, qn, W, h, d = 21, 8, 5, 3, 16
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(qn, ctx)], h, h, d)
    out = _attn(q, kp, vp, ql, cl, bt, h, h, 0.25, window=W)
    K = pa.gather_logical(kp, bt[0], ctx, P)
    V = pa.gather_logical(vp, bt[0], ctx, P)
    pos = torch.arange(ctx - qn, ctx)[:, None]
    key = torch.arange(ctx)[None, :]
    mask = (key <= pos) & (key > pos - W)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), torch.from_numpy(K).permute(1, 0, 2),
        torch.from_numpy(V).permute(1, 0, 2), attn_mask=mask, scale=0.25).permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def test_window_reads_no_page_below_it():
    """Pages holding no key inside any row's window are never looked up: an
    invalid block-table entry there changes nothing."""
    rng = np.random.default_rng(114)
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(1, 30), (3, 27)], 2, 2, 8)
    W = 9
    ref = _attn(q, kp, vp, ql, cl, bt, 2, 2, 0.4, window=W)
    bt2 = bt.copy()
    bt2[0, :(30 - W) // P] = -999999        # row 0 sees keys 21 .. 29
    bt2[1, :(24 - W + 1) // P] = -999999    # row 1's first query (24) sees 16 ..
    np.testing.assert_array_equal(_attn(q, kp, vp, ql, cl, bt2, 2, 2, 0.4, window=W), ref)


def test_pin_catches_window_off_by_one(monkeypatch):
    """A window one key too narrow breaks the brute-force pin."""
    rng = np.random.default_rng(115)
    q, kp, vp, ql, cl, bt = _random_batch(rng, [(4, 13)], 2, 2, 8)
    ref = np.array(attention_bruteforce(q, kp, vp, ql, cl, bt, P, 2, 2, 0.5, window=5))

    def narrow(keys, pos, window=0):
        keys = np.asarray(keys)[None, :]
        pos = np.asarray(pos)[:, None]
        return (keys <= pos) & (keys > pos - window + 1)
    monkeypatch.setattr(pa, "visible_mask", narrow)
    out = _attn(q, kp, vp, ql, cl, bt, 2, 2, 0.5, window=5)
    assert not np.allclose(out, ref, atol=1e-6)
