"""GPU-test helpers: run one hybrid-batch step through the C ABI and compute
the oracle's answer for the same seeded inputs."""
import math
import os

import numpy as np
import torch

from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from chunked_prefill_decode_gb300.device import device_batch
from oracle import paged_attention as pa

bits = workloads.bf16_bits
MAX_ABS, MEAN_ABS = 1e-2, 1e-3


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def gpu_step(layout, ten, scale=None, repeats=1, check=True, new_kv=False):
    """Append + plan + attention on cuda:0 (new_kv: hb_attention_new_kv, which
    reads the chunks' new rows from k_new / v_new).  Returns (k_cache,
    v_cache, out) as device tensors (the caches after append)."""
    hb = lib()
    sh = layout.shape
    scale = scale if scale is not None else 1.0 / math.sqrt(sh.head_dim)
    dev = torch.device("cuda:0")
    db = device_batch(layout.q_len, layout.context_len, layout.block_table,
                      layout.num_pages, sh.num_q_heads, sh.num_kv_heads, sh.head_dim,
                      sh.page_size, dev, sliding_window=sh.sliding_window)
    q, kn, vn = (t.to(dev) for t in (ten.q, ten.k_new, ten.v_new))
    kc, vc = ten.k_cache.to(dev).clone(), ten.v_cache.to(dev).clone()
    out = torch.full_like(q, float("nan"))
    hb.hb_kv_append(db.batch, kn, vn, kc, vc)
    plan, ws = hb.hb_plan(db.batch, db.q_len, db.context_len, sms())
    for _ in range(repeats):
        if new_kv:
            hb.hb_attention_new_kv(db.batch, plan, q, kn, vn, kc, vc, scale, out, ws)
        else:
            hb.hb_attention(db.batch, plan, q, kc, vc, scale, out, ws)
    if check:
        hb.hb_check()
    torch.cuda.synchronize()
    return kc, vc, out


def oracle_step(layout, ten, scale=None, tokens=None):
    sh = layout.shape
    scale = scale if scale is not None else 1.0 / math.sqrt(sh.head_dim)
    kp, vp = pa.kv_append(bits(ten.k_cache), bits(ten.v_cache), bits(ten.k_new),
                          bits(ten.v_new), layout.q_len, layout.context_len,
                          layout.block_table, sh.page_size)
    ref = pa.attention(bits(ten.q), kp, vp, layout.q_len, layout.context_len,
                       layout.block_table, sh.page_size, sh.num_q_heads,
                       sh.num_kv_heads, scale, tokens=tokens, window=sh.sliding_window)
    return kp, vp, ref


# (test id, max-abs error, mean-abs error, and both beyond the exact answer's
# own bf16 rounding) of every compare() in this process, reported at the end
# of the run (conftest.py) so the margin to the bounds is visible before a
# regression reaches them
MARGINS = []


def compare(out, ref, tokens=None, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = out.float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        got, ref = got[tokens], ref[tokens]
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref)
    # the exact answer's own bf16 rounding: no bf16 output can do better
    floor = np.abs(torch.from_numpy(np.asarray(ref, np.float32)).to(torch.bfloat16)
                   .double().numpy() - ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    MARGINS.append((test, float(err.max()), float(err.mean()), float((err - floor).max()),
                    float(err.mean() - floor.mean())))
    assert err.max() <= max_abs and err.mean() <= mean_abs, \
        f"max-abs {err.max():.3e} mean-abs {err.mean():.3e}"
    return err.max(), err.mean()


def compact_layout(layout, ten_dev, seqs):
    """Host copy of just the pages of `seqs` (pre-append pools), renumbered,
    so the oracle can run on a full-size batch's selected sequences."""
    sh = layout.shape
    P = sh.page_size
    pages = []
    for s in seqs:
        n = -(-int(layout.context_len[s]) // P)
        pages.extend(int(p) for p in layout.block_table[s, :n])
    pages = sorted(set(pages))
    remap = {p: i for i, p in enumerate(pages)}
    idx = torch.tensor(pages, dtype=torch.long, device=ten_dev.k_cache.device)
    kc = ten_dev.k_cache.index_select(0, idx).cpu()
    vc = ten_dev.v_cache.index_select(0, idx).cpu()
    cu = layout.cu_q_len
    rows = [(int(layout.q_len[s]), int(layout.context_len[s])) for s in seqs]
    maxp = max(-(-c // P) for _, c in rows)
    bt = np.full((len(seqs), maxp), -1, np.int32)
    for i, s in enumerate(seqs):
        n = -(-int(layout.context_len[s]) // P)
        bt[i, :n] = [remap[int(p)] for p in layout.block_table[s, :n]]
    tok = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])
    tok_t = torch.from_numpy(tok).to(ten_dev.q.device)
    sub = workloads.BatchLayout(sh, np.array([r[0] for r in rows], np.int32),
                                np.array([r[1] for r in rows], np.int32), bt,
                                len(pages), [layout.kind[s] for s in seqs])
    sub_ten = workloads.BatchTensors(ten_dev.q.index_select(0, tok_t).cpu(),
                                     ten_dev.k_new.index_select(0, tok_t).cpu(),
                                     ten_dev.v_new.index_select(0, tok_t).cpu(), kc, vc)
    return sub, sub_ten, tok
