"""The tensor-core linear layer (hb_linear) against the fp64 oracle.

Inputs: x ~ N(0, 1), W ~ N(0, 1/K) in bf16, so outputs are O(1).  Bar: the
output is bf16 (half an ulp = 2^-9 relative) after an fp32 sum over K, so
|gpu - oracle| <= 2^-8 |oracle| + 2e-3 element-wise; rows past M and other
memory are left untouched."""
import numpy as np
import pytest
import torch

from _hbutil import lib
from chunked_prefill_decode_gb300 import workloads
from oracle import linear as ol

pytestmark = pytest.mark.gpu

RTOL, ATOL = 2.0 ** -8, 2e-3
SENT = 0x7FC1


def _rand(shape, scale, gen):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def _buf(M, cols, dev):
    """[M, cols] view into a buffer with 3 sentinel rows after it."""
    full = torch.full((M + 3, cols), SENT, dtype=torch.int16, device=dev).view(torch.bfloat16)
    return full, full[:M]


def _check(got, ref):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = RTOL * np.abs(ref) + ATOL
    assert np.isfinite(g).all()
    assert (err <= bound).all(), f"worst excess {(err - bound).max():.3e}"


def _sentinels_kept(full, M):
    assert (full[M:].view(torch.int16) == SENT).all()


# tile counts from 1 to a few waves over the SMs, ragged M everywhere
@pytest.mark.parametrize("M,cols,K", [
    (1, (256,), 64), (5, (512,), 128), (128, (256,), 4096), (200, (256, 512), 192),
    (513, (4096, 1024, 1024), 512), (2048, (1024,), 256), (130, (256, 256, 256), 64),
    (1280, (4096,), 128), (1500, (2048, 1024, 1024), 256),
])
def test_store(M, cols, K):
    hb = lib()
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(M + K)
    N = sum(cols)
    x, w = _rand((M, K), 1.0, g), _rand((N, K), K ** -0.5, g)
    bufs = [_buf(M, c, dev) for c in cols]
    hb.hb_linear(x.to(dev), w.to(dev), [b[1] for b in bufs])
    hb.hb_check()
    ref = ol.linear(workloads.bf16_bits(x), workloads.bf16_bits(w))
    c0 = 0
    for (full, view), c in zip(bufs, cols):
        _check(view, ref[:, c0:c0 + c])
        _sentinels_kept(full, M)
        c0 += c


@pytest.mark.parametrize("M,F,K", [(1, 128, 64), (300, 1024, 256), (512, 2048, 1024),
                                   (1280, 2048, 128)])
def test_gated(M, F, K):
    hb = lib()
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(7 * M + F)
    x, w = _rand((M, K), 1.0, g), _rand((2 * F, K), K ** -0.5, g)
    full, view = _buf(M, F, dev)
    hb.hb_linear(x.to(dev), w.to(dev), [view], epilogue=hb.LINEAR_GATED)
    hb.hb_check()
    ref = ol.gated_mlp_up(workloads.bf16_bits(x), workloads.bf16_bits(w))
    _check(view, ref)
    _sentinels_kept(full, M)


@pytest.mark.parametrize("M,N,K", [(77, 512, 128), (640, 256, 2048), (1280, 4096, 64)])
def test_residual(M, N, K):
    hb = lib()
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(11 * M + N)
    x, w, y0 = _rand((M, K), 1.0, g), _rand((N, K), K ** -0.5, g), _rand((M, N), 1.0, g)
    full, view = _buf(M, N, dev)
    view.copy_(y0.to(dev))
    hb.hb_linear(x.to(dev), w.to(dev), [view], epilogue=hb.LINEAR_RESIDUAL)
    hb.hb_check()
    ref = ol.residual(workloads.bf16_bits(y0), workloads.bf16_bits(x), workloads.bf16_bits(w))
    _check(view, ref)
    _sentinels_kept(full, M)


def test_repeated_launches_and_timing():
    hb = lib()
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(3)
    x, w = _rand((384, 512), 1.0, g).to(dev), _rand((1024, 512), 512 ** -0.5, g).to(dev)
    y = torch.empty(384, 1024, dtype=torch.bfloat16, device=dev)
    hb.hb_timing_enable(True)
    for _ in range(5):
        hb.hb_linear(x, w, [y])
    t = hb.hb_timing_read()
    hb.hb_timing_enable(False)
    hb.hb_check()
    assert t["linear"][1] == 5 and t["linear"][0] > 0
    ref = ol.linear(workloads.bf16_bits(x.cpu()), workloads.bf16_bits(w.cpu()))
    _check(y, ref)


@pytest.mark.parametrize("M,N,K,epi", [(1, 256, 4096, 0), (200, 512, 4096, 0), (77, 512, 2048, 2),
                                       (300, 512, 1024, 1), (256, 4096, 14336, 0)])
def test_split_k_matches_unsplit(M, N, K, epi):
    """Few tiles: the K range is split over CTAs (workspace given) -- same bar
    as the unsplit kernel, and repeated calls reuse the workspace."""
    hb = lib()
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(M + N + K)
    x, w = _rand((M, K), 1.0, g).to(dev), _rand((N, K), K ** -0.5, g).to(dev)
    cols = N // 2 if epi == 1 else N
    y0 = _rand((M, cols), 1.0, g).to(dev)
    assert hb.linear_workspace(M, N, K, epi, dev) is not None
    outs = {}
    for ws in ("auto", None):
        y = y0.clone()
        for _ in range(2 if epi != 2 else 1):
            hb.hb_linear(x, w, [y], epilogue=epi, workspace=ws)
        hb.hb_check()
        outs[ws] = y
    xb, wb = workloads.bf16_bits(x.cpu()), workloads.bf16_bits(w.cpu())
    if epi == 0:
        ref = ol.linear(xb, wb)
    elif epi == 1:
        ref = ol.gated_mlp_up(xb, wb)
    else:
        ref = ol.residual(workloads.bf16_bits(y0.cpu()), xb, wb)
    _check(outs["auto"], ref)
    _check(outs[None], ref)


def test_one_workspace_serves_every_shape():
    """The cached workspace is shared by problems of different shapes (the
    counters sit at a fixed place): interleaved calls all meet the bar."""
    hb = lib()
    dev = torch.device("cuda:0")
    g = torch.Generator().manual_seed(99)
    shapes = [(1, 256, 4096), (300, 1024, 2048), (64, 512, 8192), (1, 256, 4096), (200, 768, 512)]
    for M, N, K in shapes * 2:
        x, w = _rand((M, K), 1.0, g).to(dev), _rand((N, K), K ** -0.5, g).to(dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        hb.hb_linear(x, w, [y])
        hb.hb_check()
        _check(y, ol.linear(workloads.bf16_bits(x.cpu()), workloads.bf16_bits(w.cpu())))
