"""Oracle for the linear layers around the attention step (fp64, CPU).

TEST INFRASTRUCTURE, like the rest of `oracle/`: only `tests/`,
`__graft_entry__.smoke()` and `bench.py`'s CPU legs may import it; it shares
no code with the CUDA library.

"Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
延迟权衡", §问题背景 (两阶段天然不对称): a hybrid batch's tokens also pass
through the model's linear layers, which take most of the time of both
phases -- compute-bound for prefill tokens, bound by reading the weights for
decode tokens.  The pages do not write the layers out; the readings taken
are the plain ones of a GQA transformer block:
  * a linear layer is y = x W^T, x [M, K] (one row per token of the batch),
    W [N, K] (row n holds the weights of output feature n);
  * the gated MLP multiplies silu(x W_gate^T) with x W_up^T elementwise,
    silu(g) = g / (1 + e^-g), with W_gate and W_up stacked as one [2F, K]
    weight (gate rows first);
  * residual connections add a layer's output to its input stream.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import bf16_to_f64


def _f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(np.float64)


def linear(x, w) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * w[n, k], in float64."""
    x, w = _f64(x), _f64(w)
    if x.ndim != 2 or w.ndim != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x [M, K] and w [N, K] needed")
    return x @ w.T


def silu(g) -> np.ndarray:
    """g * sigmoid(g) = g / (1 + exp(-g)), written to stay finite for large |g|."""
    g = np.asarray(g, dtype=np.float64)
    return np.where(g >= 0, g / (1.0 + np.exp(-np.abs(g))),
                    g * np.exp(-np.abs(g)) / (1.0 + np.exp(-np.abs(g))))


def gated_mlp_up(x, w_gate_up) -> np.ndarray:
    """silu(x W_gate^T) * (x W_up^T) for W = [W_gate; W_up] of shape [2F, K]."""
    w = _f64(w_gate_up)
    if w.shape[0] % 2:
        raise ValueError("stacked gate/up weight needs an even row count")
    f = w.shape[0] // 2
    return silu(linear(x, w[:f])) * linear(x, w[f:])


def residual(y_in, x, w) -> np.ndarray:
    """y_in + x W^T."""
    return _f64(y_in) + linear(x, w)
