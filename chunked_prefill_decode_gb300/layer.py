"""One transformer block of a hybrid batch: the linear layers around the
attention step, every step in this library's kernels.

"Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
延迟权衡", §问题背景 (两阶段天然不对称): besides attention, every token of a
hybrid batch passes through the model's linear layers, which take most of
the iteration; chunking a prefill lets its tokens share those weight reads
with the decode tokens of the same iteration.  The pages do not write the
block out; the plain GQA block is taken (norms and rotary embeddings, which
are elementwise and outside the pages, are left out):

    q, k, v = split(x Wqkv^T)                    hb_linear, split epilogue
    append k, v to the paged cache               hb_kv_append
    a = attention(q, cache)                       hb_plan + hb_attention_new_kv
    x = x + a Wo^T                                hb_linear, residual epilogue
    m = silu(x Wg^T) * (x Wu^T)                   hb_linear, gated epilogue
    x = x + m Wd^T                                hb_linear, residual epilogue

Weights are synthetic (seeded, N(0, 1/fan_in) in bf16): no trained weights
are needed to time or check the block.  The residual stream x is updated in
place.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from . import hb


@dataclass
class BlockShape:
    hidden: int = 4096          # model width H
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 14336            # gated-MLP width F
    page_size: int = 16

    @property
    def q_cols(self):
        return self.num_q_heads * self.head_dim

    @property
    def kv_cols(self):
        return self.num_kv_heads * self.head_dim

    def params(self) -> int:
        H = self.hidden
        return (self.q_cols + 2 * self.kv_cols) * H + H * self.q_cols + 2 * self.ffn * H + H * self.ffn


MISTRAL_7B = BlockShape()
YI_34B = BlockShape(hidden=7168, num_q_heads=56, num_kv_heads=8, head_dim=128, ffn=20480)


class HybridBlock:
    """Synthetic weights of one block on a device, and its forward step."""

    def __init__(self, shape: BlockShape = MISTRAL_7B, seed: int = 0, device="cuda"):
        s = shape
        for name, v in (("hidden", s.hidden), ("q columns", s.q_cols), ("kv columns", s.kv_cols),
                        ("ffn", s.ffn)):
            if v % 256:
                raise ValueError(f"{name} ({v}) must be a multiple of 256 for the GEMM tiles")
        self.shape = s
        self.dev = torch.device(device)
        g = torch.Generator(device=self.dev).manual_seed(seed)

        def weight(n, k):
            return (torch.randn(n, k, generator=g, device=self.dev) / math.sqrt(k)).to(torch.bfloat16)
        H = s.hidden
        self.w_qkv = weight(s.q_cols + 2 * s.kv_cols, H)
        self.w_o = weight(H, s.q_cols)
        self.w_gu = weight(2 * s.ffn, H)
        self.w_d = weight(H, s.ffn)
        self.scale = 1.0 / math.sqrt(s.head_dim)
        self._plan = None
        self._ws = None
        self._sms = torch.cuda.get_device_properties(self.dev).multi_processor_count

    def buffers(self, tokens: int) -> dict:
        """Activation buffers for a batch of `tokens` new tokens."""
        s = self.shape
        e = dict(dtype=torch.bfloat16, device=self.dev)
        return {"q": torch.empty(tokens, s.q_cols, **e),
                "k": torch.empty(tokens, s.kv_cols, **e),
                "v": torch.empty(tokens, s.kv_cols, **e),
                "a": torch.empty(tokens, s.q_cols, **e),
                "m": torch.empty(tokens, s.ffn, **e)}

    def forward(self, x, batch, k_cache, v_cache, bufs=None, plan=True, snapshot=False):
        """x: [T, H] bf16 residual stream (updated in place); batch: an
        hb_batch (device.device_batch) of the same T new tokens; k_cache,
        v_cache: the layer's page pools.  Returns the buffers used; with
        snapshot=True they also hold a copy of the residual stream after the
        attention block ("h", for checking the stages one by one)."""
        T = x.shape[0]
        b = bufs if bufs is not None else self.buffers(T)
        hb.hb_linear(x, self.w_qkv, [b["q"], b["k"], b["v"]])
        hb.hb_kv_append(batch.batch, b["k"], b["v"], k_cache, v_cache)
        if plan or self._plan is None:
            self._plan, self._ws = hb.hb_plan(batch.batch, batch.q_len, batch.context_len,
                                              self._sms, workspace=self._ws, plan=self._plan)
        hb.hb_attention_new_kv(batch.batch, self._plan, b["q"], b["k"], b["v"], k_cache, v_cache,
                               self.scale, b["a"], self._ws)
        hb.hb_linear(b["a"], self.w_o, [x], epilogue=hb.LINEAR_RESIDUAL)
        if snapshot:
            b["h"] = x.clone()
        hb.hb_linear(x, self.w_gu, [b["m"]], epilogue=hb.LINEAR_GATED)
        hb.hb_linear(b["m"], self.w_d, [x], epilogue=hb.LINEAR_RESIDUAL)
        return b

    def flops(self, tokens: int) -> float:
        """Linear-layer FLOPs of the block for `tokens` new tokens."""
        return 2.0 * self.shape.params() * tokens
