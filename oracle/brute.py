"""Pure-Python brute force of the paged hybrid-batch attention (tiny shapes).

TEST INFRASTRUCTURE: a second, loop-by-loop statement of the same definition
as oracle.paged_attention.attention, written with Python floats, math.exp and
explicit index arithmetic through the block table, so the numpy oracle can be
checked against something that shares none of its array code.  Only `tests/`
use it.  Definition followed: "Sarathi-Serve：以 chunked-prefills 与 stall-free
batching 驯服 LLM 推理的吞吐—延迟权衡", §GPU / 系统数据路径 ⑤ (attention over
the KV cache read through the page table), with the causal, absolute-position
mask reading stated in oracle.paged_attention.
"""
from __future__ import annotations

import math


def _val(x):
    return float(x)


def attention_bruteforce(q, k_pool, v_pool, q_len, context_len, block_table,
                         page_size, num_q_heads, num_kv_heads, scale, window=0):
    """Nested-loop attention; q, pools are float64 arrays; returns a list
    out[token][head][d] of Python floats.  With window > 0 the query at p
    sees keys p - window + 1 .. p only ("Sarathi-Serve: Chunked Prefills for
    Stall-Free LLM Inference", §Results and evidence, names such variants)."""
    g = num_q_heads // num_kv_heads
    D = len(q[0][0])
    out = []
    start = 0
    for s in range(len(q_len)):
        ql = int(q_len[s])
        ctx = int(context_len[s])
        for j in range(ql):
            p = ctx - ql + j
            first = max(0, p - window + 1) if window > 0 else 0
            keys = list(range(first, p + 1))
            row = []
            for h in range(num_q_heads):
                kv = h // g
                scores = []
                for t in keys:
                    page = int(block_table[s][t // page_size])
                    slot = t % page_size
                    acc = 0.0
                    for d in range(D):
                        acc += _val(q[start + j][h][d]) * _val(k_pool[page][slot][kv][d])
                    scores.append(scale * acc)
                mx = max(scores)
                w = [math.exp(x - mx) for x in scores]
                z = sum(w)
                o = []
                for d in range(D):
                    acc = 0.0
                    for i, t in enumerate(keys):
                        page = int(block_table[s][t // page_size])
                        acc += w[i] * _val(v_pool[page][t % page_size][kv][d])
                    o.append(acc / z)
                row.append(o)
            out.append(row)
        start += ql
    return out
