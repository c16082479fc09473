"""Oracle for the hybrid-batch attention step over a paged KV cache (fp64, CPU).

TEST INFRASTRUCTURE.  This module states what the CUDA path must compute, in
the plainest form: numpy in float64, one sequence and one head at a time, no
tiling, no fusion, no split of the keys, no online softmax.  Only `tests/`,
`__graft_entry__.smoke()` and `bench.py`'s CPU-baseline / reference leg may
import it; the product path never does, and it shares no code with the CUDA
library (its only inputs are arrays handed to it).

What the pages fix, and where:
  * "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的
    吞吐—延迟权衡", §GPU / 系统数据路径 ⑤: attention reads and writes the KV cache
    through the PagedAttention page table; a prefill chunk appends its new KV,
    a decode reads all earlier KV, and chunk i re-reads the KV of the earlier
    chunks of its prompt.
  * same page, §核心机制 3: splitting a prefill into N chunks adds KV re-reads
    but leaves the amount of computation unchanged -- chunking changes cost,
    not the result.
  * "Sarathi-Serve: Chunked Prefills for Stall-Free LLM Inference", "What to
    notice when reading": every prompt token is still paid for, only spread
    over iterations.
  * "In-flight Batching", §KV Cache 管理的协同优化: fixed 16-token pages, a block
    table maps logical pages to physical ones, which need not be contiguous.

Readings taken where the pages are silent:
  * attention is standard scaled dot-product attention with a causal mask
    aligned to absolute positions: the new token j of a row with q_len new
    tokens and context_len cached-after-append tokens sits at position
    p = context_len - q_len + j and sees keys 0..p;
  * grouped-query attention maps q head h to kv head h // (Hq / Hkv);
  * pages are laid out [page][slot][kv_head][head_dim], separate K and V pools;
    the oracle only ever looks at the logical view through the block table;
  * "Sarathi-Serve: Chunked Prefills for Stall-Free LLM Inference", §Results
    and evidence, names sliding-window model variants without a size: with a
    window of W tokens the query at position p sees keys p - W + 1 .. p (W
    keys, itself included); W = 0 means no window.

Parity pins (tests/test_oracle_pins.py) tie this module to things other than
itself: a pure-Python brute force, closed forms (constant V, q = 0, one key,
two keys), chunked == unchunked, decode row == last prefill row, causality,
physical-page permutation invariance, GQA == expanded MHA, and torch's fp64
scaled_dot_product_attention with an explicit bottom-right causal mask.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns: a bf16 is the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def _as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(np.float64)


def _cu(q_len) -> np.ndarray:
    q_len = np.asarray(q_len, dtype=np.int64)
    cu = np.zeros(q_len.shape[0] + 1, dtype=np.int64)
    np.cumsum(q_len, out=cu[1:])
    return cu


def new_token_positions(q_len_s: int, context_len_s: int) -> np.ndarray:
    """Logical positions of a row's new tokens: the q_len most recent ones."""
    return np.arange(context_len_s - q_len_s, context_len_s, dtype=np.int64)


def query_positions(q_len_s: int, context_len_s: int) -> np.ndarray:
    """Absolute position of each query row of a sequence (what the causal
    mask compares key indices with): bottom-right aligned, the last query is
    the newest token, at context_len - 1."""
    return context_len_s - q_len_s + np.arange(q_len_s, dtype=np.int64)


def kv_append(k_pool, v_pool, k_new, v_new, q_len, context_len, block_table,
              page_size):
    """Scatter every new token's K and V rows into its page slot.

    New token j of sequence s sits at logical position
    pos = context_len[s] - q_len[s] + j and goes to physical page
    block_table[s][pos // page_size], slot pos % page_size.  The copy is of
    raw values (bit patterns), so any dtype works; returns new pools.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    cu = _cu(q_len)
    for s in range(len(q_len)):
        pos = new_token_positions(int(q_len[s]), int(context_len[s]))
        pages = np.asarray(block_table)[s, pos // page_size]
        slots = pos % page_size
        rows = slice(int(cu[s]), int(cu[s + 1]))
        k_out[pages, slots] = np.asarray(k_new)[rows]
        v_out[pages, slots] = np.asarray(v_new)[rows]
    return k_out, v_out


def gather_logical(pool, block_table_row, n_tokens, page_size, start=0) -> np.ndarray:
    """Tokens start .. n_tokens-1 of one sequence, in logical order: [n, Hkv, D]."""
    pos = np.arange(start, n_tokens, dtype=np.int64)
    return np.asarray(pool)[np.asarray(block_table_row)[pos // page_size],
                            pos % page_size]


def visible_mask(keys, pos, window=0) -> np.ndarray:
    """[n, K] bool: key position keys[k] is visible to the query at position
    pos[i] -- causal (key <= query) and, with a sliding window of W tokens,
    no more than W - 1 positions back."""
    keys = np.asarray(keys, dtype=np.int64)[None, :]
    pos = np.asarray(pos, dtype=np.int64)[:, None]
    vis = keys <= pos
    if window > 0:
        vis &= keys > pos - window
    return vis


def attention(q, k_pool, v_pool, q_len, context_len, block_table, page_size,
              num_q_heads, num_kv_heads, scale, tokens=None, window=0) -> np.ndarray:
    """fp64 output [T, Hq, D] of the hybrid batch's attention.

    For sequence s, new token j, q head h (kv head h // g, g = Hq / Hkv):
        p    = context_len[s] - q_len[s] + j
        s_t  = scale * <q[s, j, h], K[t, kv]>            for t = t0 .. p
        o    = sum_t softmax(s)_t * V[t, kv]
    with t0 = 0, or t0 = max(0, p - window + 1) with a sliding window, and K,
    V read through the block table after the append (only the pages holding
    keys some query sees).  `tokens`, if given, restricts the computation to
    those global token indices (other rows of the result are NaN), for spot
    checks of large batches.
    """
    qf = _as_f64(q)
    T, Hq, D = qf.shape
    if Hq != num_q_heads or num_q_heads % num_kv_heads:
        raise ValueError("bad head counts")
    g = num_q_heads // num_kv_heads
    out = np.full((T, Hq, D), np.nan)
    want = None if tokens is None else set(int(t) for t in tokens)
    cu = _cu(q_len)
    for s in range(len(q_len)):
        ql, ctx = int(q_len[s]), int(context_len[s])
        rows = np.arange(int(cu[s]), int(cu[s + 1]))
        if want is not None:
            sel = np.array([r in want for r in rows], dtype=bool)
            if not sel.any():
                continue
        else:
            sel = np.ones(ql, dtype=bool)
        pos = query_positions(ql, ctx)[sel]                  # [n]
        t0 = max(0, int(pos.min()) - window + 1) if window > 0 else 0
        K = _as_f64(gather_logical(k_pool, block_table[s], ctx, page_size, t0))
        V = _as_f64(gather_logical(v_pool, block_table[s], ctx, page_size, t0))
        visible = visible_mask(np.arange(t0, ctx), pos, window)   # [n, ctx - t0]
        for h in range(Hq):
            kv = h // g
            scores = scale * (qf[rows[sel], h, :] @ K[:, kv, :].T)
            scores = np.where(visible, scores, -np.inf)
            m = scores.max(axis=1, keepdims=True)
            w = np.exp(scores - m)
            w /= w.sum(axis=1, keepdims=True)
            out[rows[sel], h, :] = w @ V[:, kv, :]
    return out


def partial_softmax_state(scores, values):
    """(m, l, o) of one key range: m = max score, l = sum exp(s - m),
    o = sum exp(s - m) * v (unnormalised).  Used by the merge pin."""
    scores = np.asarray(scores, dtype=np.float64)
    m = scores.max()
    w = np.exp(scores - m)
    return m, w.sum(), w @ np.asarray(values, dtype=np.float64)


def merge_partial_states(states):
    """Combine the (m, l, o) of disjoint key ranges into the softmax output.

    m = max_i m_i;  l = sum_i exp(m_i - m) l_i;  o = sum_i exp(m_i - m) o_i / l.
    This is the usual way to join softmaxes of split key ranges; the pages do
    not describe it (it is the split-KV merge the CUDA path uses)."""
    m = max(st[0] for st in states)
    l = sum(np.exp(st[0] - m) * st[1] for st in states)
    o = sum(np.exp(st[0] - m) * st[2] for st in states)
    return o / l
