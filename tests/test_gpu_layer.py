"""One transformer block of a hybrid batch (layer.HybridBlock) in this
library's kernels, checked stage by stage against the fp64 oracle fed with
the GPU's own bf16 intermediates: each stage within its own bar (linear
layers: 2^-8 relative + 2e-3; attention: max-abs 1e-2, mean-abs 1e-3; the
append bit-exact)."""
import math

import numpy as np
import pytest
import torch

from _gpu import compare
from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from chunked_prefill_decode_gb300.device import from_layout
from chunked_prefill_decode_gb300.layer import BlockShape, HybridBlock
from chunked_prefill_decode_gb300.workloads import Shape, layout_from_rows
from oracle import linear as ol
from oracle import paged_attention as pa

pytestmark = pytest.mark.gpu
bits = workloads.bf16_bits


def _close(got, ref, rtol=2.0 ** -8, atol=2e-3):
    g = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    excess = np.abs(g - ref) - (rtol * np.abs(ref) + atol)
    assert (excess <= 0).all(), f"worst excess {excess.max():.3e}"


@pytest.mark.parametrize("hq,hkv,window", [(8, 2, 0), (16, 2, 0), (8, 2, 40)])
def test_block_stage_by_stage(hq, hkv, window):
    lib()
    bs = BlockShape(hidden=512, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, ffn=1024)
    blk = HybridBlock(bs, seed=hq + window)
    rows = [(1, 300), (1, 41), (70, 70), (1, 129), (33, 600)]
    lay = layout_from_rows(Shape(hq, hkv, 128, sliding_window=window), rows, 21)
    ten = workloads.make_tensors(lay, 21, device="cuda")      # pools (q, k_new unused)
    db = from_layout(lay)
    T = lay.total_q
    g = torch.Generator(device="cuda").manual_seed(5)
    x0 = torch.randn(T, bs.hidden, generator=g, device="cuda").to(torch.bfloat16)
    x = x0.clone()
    kc, vc = ten.k_cache.clone(), ten.v_cache.clone()
    b = blk.forward(x, db, kc, vc, snapshot=True)
    torch.cuda.synchronize()
    lib().hb_check()
    # QKV projection, split over three outputs
    qkv = ol.linear(bits(x0), bits(blk.w_qkv))
    _close(b["q"], qkv[:, :bs.q_cols])
    _close(b["k"], qkv[:, bs.q_cols:bs.q_cols + bs.kv_cols])
    _close(b["v"], qkv[:, bs.q_cols + bs.kv_cols:])
    # append (bit-exact) and attention of the GPU's own q, k, v
    kp, vp = pa.kv_append(bits(ten.k_cache), bits(ten.v_cache),
                          bits(b["k"]).reshape(T, hkv, 128), bits(b["v"]).reshape(T, hkv, 128),
                          lay.q_len, lay.context_len, lay.block_table, 16)
    assert np.array_equal(bits(kc), kp) and np.array_equal(bits(vc), vp)
    att = pa.attention(bits(b["q"]).reshape(T, hq, 128), kp, vp, lay.q_len, lay.context_len,
                       lay.block_table, 16, hq, hkv, 1 / math.sqrt(128), window=window)
    compare(b["a"].view(T, hq, 128), att)
    # output projection into the residual stream, gated MLP, down projection
    _close(b["h"], ol.residual(bits(x0), bits(b["a"]), bits(blk.w_o)))
    _close(b["m"], ol.gated_mlp_up(bits(b["h"]), bits(blk.w_gu)))
    _close(x, ol.residual(bits(b["h"]), bits(b["m"]), bits(blk.w_d)))
