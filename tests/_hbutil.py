"""Shared test helpers: build/load the library, fake host-only batches."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_built = False


def lib():
    """Build (if stale) and load libhb.so."""
    global _built
    from chunked_prefill_decode_gb300 import hb
    if not _built:
        from chunked_prefill_decode_gb300.build import build
        build()
        _built = True
    hb.load()
    return hb


def header_functions():
    """Names of the functions include/hb.h declares."""
    with open(os.path.join(ROOT, "include", "hb.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(hb_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def host_batch(hb, rows, hq=32, hkv=8, d=128, max_pages=None, num_pages=None, window=0):
    """hb_batch with fake (never dereferenced) device pointers, for host-only
    calls such as hb_plan without a workspace."""
    import numpy as np
    ql = np.array([r[0] for r in rows], np.int32)
    cl = np.array([r[1] for r in rows], np.int32)
    mp = max_pages or max(1, max(-(-c // 16) for c in cl)) if len(rows) else 1
    npg = num_pages or max(1, int(sum(-(-c // 16) for c in cl)))
    fake = 0x1000
    b = hb.make_batch(len(rows), int(ql.sum()), mp, npg, hq, hkv, d,
                      None, None, None, sliding_window=window)
    if len(rows):
        b.cu_q_len = b.context_len = b.block_table = fake
    return b, ql, cl
