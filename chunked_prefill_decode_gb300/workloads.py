"""Seeded synthetic hybrid batches (inputs only; none of the method's arithmetic).

This module is the one place that both the CPU oracle's tests and the CUDA path
draw their inputs from.  It builds *shapes* and *random values*: the list of
rows of one hybrid batch (decode rows with q_len = 1 plus prefill chunks), a
block table that maps each sequence's logical pages onto a seeded random
permutation of physical pages, and bf16 tensors drawn from N(0, 1).  It never
computes attention, never scatters KV into pages and never schedules requests.

Shapes follow the workloads the Sarathi-Serve pages describe:
  * "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的
    吞吐—延迟权衡", §3 分钟速读 item 4 and §测试床与负载: prompt/output medians
    1730/415 (openchat_sharegpt4) and 7059/208 (arxiv_summarization), totals
    truncated at 8192 / 16384, budgets 512 (strict) and 2048 (relaxed).
  * "In-flight Batching", §KV Cache 管理的协同优化: 16-token pages mapped by a
    block table, physical pages need not be contiguous.
The traces themselves are not available; lognormal stand-ins with those
medians (sigma 0.6) replace them.

A row is described by (q_len, context_len): context_len counts the tokens in
the cache *after* this step's new tokens are appended, so the row's new tokens
sit at logical positions context_len - q_len .. context_len - 1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_SIZE = 16
# bf16 quiet-NaN bit pattern used to poison every pool slot that holds no
# cached token: a kernel that reads past a sequence's context shows up as NaN.
SENTINEL_BITS = 0x7FC1


@dataclass
class Shape:
    """Head geometry of one attention layer (sliding_window 0: full causal;
    W > 0: a query at position p sees keys p - W + 1 .. p)."""
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int = PAGE_SIZE
    sliding_window: int = 0


@dataclass
class BatchLayout:
    """Row structure of one hybrid batch: host int32 descriptors only."""
    shape: Shape
    q_len: np.ndarray            # [S] int32
    context_len: np.ndarray      # [S] int32, after append
    block_table: np.ndarray      # [S, max_pages] int32 (unused entries = -1)
    num_pages: int               # physical pages in the pool
    kind: list = field(default_factory=list)   # "decode" | "chunk" per row

    @property
    def num_seqs(self) -> int:
        return int(self.q_len.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.q_len.sum())

    @property
    def cu_q_len(self) -> np.ndarray:
        cu = np.zeros(self.num_seqs + 1, dtype=np.int32)
        np.cumsum(self.q_len, out=cu[1:])
        return cu

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])


def _lognormal_int(rng, median, sigma, lo, hi, n):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def layout_from_rows(shape: Shape, rows, seed: int, kinds=None,
                     pool_slack: float = 0.10, min_extra_pages: int = 4,
                     max_pages_per_seq: int | None = None) -> BatchLayout:
    """Place rows [(q_len, context_len), ...] onto a seeded page permutation.

    The pool holds sum(ceil(ctx / page)) pages plus `pool_slack` spare ones;
    each sequence receives the next pages of a seeded random permutation, so
    its pages are scattered over the pool.
    """
    rng = np.random.default_rng(seed + 7919)
    P = shape.page_size
    rows = [(int(q), int(c)) for q, c in rows]
    for q, c in rows:
        if not (1 <= q <= c):
            raise ValueError(f"row needs 1 <= q_len <= context_len, got {(q, c)}")
    pages = [-(-c // P) for _, c in rows]
    used = int(sum(pages))
    num_pages = used + max(min_extra_pages, int(math.ceil(used * pool_slack)))
    perm = rng.permutation(num_pages).astype(np.int32)
    maxp = max(pages) if pages else 1
    if max_pages_per_seq is not None:
        if max_pages_per_seq < maxp:
            raise ValueError("max_pages_per_seq smaller than the longest sequence")
        maxp = max_pages_per_seq
    bt = np.full((len(rows), maxp), -1, dtype=np.int32)
    k = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[k:k + n]
        k += n
    q_len = np.array([q for q, _ in rows], dtype=np.int32)
    ctx = np.array([c for _, c in rows], dtype=np.int32)
    if kinds is None:
        kinds = ["decode" if q == 1 else "chunk" for q, _ in rows]
    return BatchLayout(shape, q_len, ctx, bt, num_pages, list(kinds))


# ---------------------------------------------------------------------------
# The benchmark workloads (one hybrid batch each).
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> BatchLayout:
    """1 layer, 8 q = 8 kv heads, head_dim 64: 4 decode rows with context
    U[100, 300] plus a 64-token chunk at offset 64 of a 128-token prompt."""
    rng = np.random.default_rng(seed)
    shape = Shape(8, 8, 64)
    rows = [(1, int(c)) for c in rng.integers(100, 301, size=4)]
    rows.append((64, 128))
    return layout_from_rows(shape, rows, seed)


def mistral_b512(seed: int = 1) -> BatchLayout:
    """Mistral-7B attention shape (32 q / 8 kv heads, head_dim 128), budget 512:
    64 decode rows with context ~ lognormal(median 2145 = 1730 + 415) clipped
    to [128, 8192], plus one 448-token chunk at a seeded chunk index k of a
    lognormal prompt (median 1730) clipped to [448, 8192]."""
    rng = np.random.default_rng(seed)
    shape = Shape(32, 8, 128)
    ctx = _lognormal_int(rng, 2145, 0.6, 128, 8192, 64)
    rows = [(1, int(c)) for c in ctx]
    c = 448
    prompt = int(_lognormal_int(rng, 1730, 0.6, c, 8192, 1)[0])
    n_full = prompt // c
    k = int(rng.integers(0, n_full))
    rows.append((c, c * (k + 1)))
    return layout_from_rows(shape, rows, seed)


def mistral_b512_window(seed: int = 1, window: int = 1024) -> BatchLayout:
    """The Mistral-7B batch of mistral_b512 with sliding-window attention of
    `window` tokens.  The pages name sliding-window variants without a size;
    1024 is below the decode rows' median context (2145), so the window
    binds for most rows."""
    lay = mistral_b512(seed)
    lay.shape = Shape(32, 8, 128, sliding_window=window)
    return lay


def yi_b2048(seed: int = 2, offset: int = 6048) -> BatchLayout:
    """Yi-34B attention shape (56 q / 8 kv heads, head_dim 128), budget 2048:
    32 decode rows with context ~ lognormal(median 7267 = 7059 + 208) clipped
    to [1, 16384], plus one 2016-token chunk at `offset` (default 6048, the
    fourth chunk of a 2016-token chunking; the prompt is taken as 8064 long)."""
    rng = np.random.default_rng(seed)
    shape = Shape(56, 8, 128)
    ctx = _lognormal_int(rng, 7267, 0.6, 1, 16384, 32)
    rows = [(1, int(c)) for c in ctx]
    rows.append((2016, offset + 2016))
    return layout_from_rows(shape, rows, seed)


def yi_b2048_o5043(seed: int = 2) -> BatchLayout:
    """The Yi-34B batch with its 2016-token chunk at offset 5043: the last
    full chunk of a 7059-token prompt (the configuration's prompt length),
    where the default takes the chunk index 3 reading of "offset ~6000"."""
    return yi_b2048(seed, offset=5043)


def decode_only(seed: int = 3) -> BatchLayout:
    """32 q / 8 kv heads, head_dim 128: 256 decode rows, context U[1024, 8192]."""
    rng = np.random.default_rng(seed)
    shape = Shape(32, 8, 128)
    rows = [(1, int(c)) for c in rng.integers(1024, 8193, size=256)]
    return layout_from_rows(shape, rows, seed)


def chunk_sweep(chunk: int, index: int | None = None, seed: int = 4,
                prompt: int = 8192, n_decode: int = 32,
                decode_ctx: int = 2048) -> BatchLayout:
    """32 q / 8 kv heads, head_dim 128: one `prompt`-token prompt prefilled in
    chunks of `chunk` tokens; this batch holds chunk number `index` (default:
    the last one) next to `n_decode` decode rows of context `decode_ctx`."""
    shape = Shape(32, 8, 128)
    n_chunks = -(-prompt // chunk)
    if index is None:
        index = n_chunks - 1
    if not (0 <= index < n_chunks):
        raise ValueError("chunk index out of range")
    off = index * chunk
    c = min(chunk, prompt - off)
    rows = [(1, decode_ctx)] * n_decode + [(c, off + c)]
    return layout_from_rows(shape, rows, seed + 1000 * chunk + index)


WORKLOADS = {
    "tiny": tiny,
    "mistral_b512": mistral_b512,
    "mistral_b512_window": mistral_b512_window,
    "yi_b2048": yi_b2048,
    "yi_b2048_o5043": yi_b2048_o5043,
    "decode_only": decode_only,
}


# ---------------------------------------------------------------------------
# Tensor contents.
# ---------------------------------------------------------------------------

@dataclass
class BatchTensors:
    """bf16 tensors of one batch (on the device of the generator)."""
    q: torch.Tensor         # [T, Hq, D]
    k_new: torch.Tensor     # [T, Hkv, D]
    v_new: torch.Tensor     # [T, Hkv, D]
    k_cache: torch.Tensor   # [num_pages, P, Hkv, D] (before append)
    v_cache: torch.Tensor


def _normal_bf16(gen, shape, device):
    return torch.randn(shape, generator=gen, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def cached_slot_mask(layout: BatchLayout) -> np.ndarray:
    """Boolean [num_pages, P]: slots holding a token cached before this step
    (logical position < context_len - q_len of the owning sequence)."""
    P = layout.shape.page_size
    mask = np.zeros((layout.num_pages, P), dtype=bool)
    for s in range(layout.num_seqs):
        n_cached = int(layout.context_len[s] - layout.q_len[s])
        for lp in range(-(-n_cached // P)):
            page = layout.block_table[s, lp]
            n = min(P, n_cached - lp * P)
            mask[page, :n] = True
    return mask


def make_tensors(layout: BatchLayout, seed: int, device="cpu") -> BatchTensors:
    """Draw q, k_new, v_new and the pre-append pools from N(0, 1) in bf16.

    Pool slots that hold no cached token (free pages, tails of last pages and
    the positions this step will append) are set to the NaN sentinel."""
    sh = layout.shape
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T = layout.total_q
    q = _normal_bf16(gen, (T, sh.num_q_heads, sh.head_dim), device)
    k_new = _normal_bf16(gen, (T, sh.num_kv_heads, sh.head_dim), device)
    v_new = _normal_bf16(gen, (T, sh.num_kv_heads, sh.head_dim), device)
    pool_shape = (layout.num_pages, sh.page_size, sh.num_kv_heads, sh.head_dim)
    k_cache = _normal_bf16(gen, pool_shape, device)
    v_cache = _normal_bf16(gen, pool_shape, device)
    hole = ~torch.from_numpy(cached_slot_mask(layout)).to(device)
    for pool in (k_cache, v_cache):
        pool.view(torch.int16).masked_fill_(hole[:, :, None, None], SENTINEL_BITS)
    return BatchTensors(q, k_new, v_new, k_cache, v_cache)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
