"""Pins of the linear-layer oracle (CPU): a pure-Python triple loop, an
identity weight, linearity, closed forms of silu, the gated MLP against its
two halves, and planted mistakes."""
import math

import numpy as np
import pytest

from oracle import linear as ol


def loops(x, w):
    """y[m][n] = sum_k x[m][k] w[n][k] with Python floats."""
    M, K = len(x), len(x[0])
    return [[sum(float(x[m][k]) * float(w[n][k]) for k in range(K)) for n in range(len(w))]
            for m in range(M)]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (4, 8, 16), (9, 2, 3)])
def test_linear_matches_loops(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x, w = rng.standard_normal((M, K)), rng.standard_normal((N, K))
    np.testing.assert_allclose(ol.linear(x, w), np.array(loops(x, w)), rtol=0, atol=1e-12)


def test_identity_weight_returns_input():
    x = np.random.default_rng(1).standard_normal((6, 8))
    np.testing.assert_array_equal(ol.linear(x, np.eye(8)), x)
    # a permutation of the identity permutes the output features
    perm = np.array([3, 0, 7, 1, 6, 2, 5, 4])
    np.testing.assert_array_equal(ol.linear(x, np.eye(8)[perm]), x[:, perm])


def test_linearity():
    rng = np.random.default_rng(2)
    x1, x2, w = rng.standard_normal((5, 12)), rng.standard_normal((5, 12)), rng.standard_normal((7, 12))
    np.testing.assert_allclose(ol.linear(x1 + 2.5 * x2, w),
                               ol.linear(x1, w) + 2.5 * ol.linear(x2, w), rtol=0, atol=1e-12)


def test_silu_closed_forms():
    assert ol.silu(0.0) == 0.0
    assert ol.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-15)
    assert ol.silu(-2.0) == pytest.approx(-2.0 / (1.0 + math.exp(2.0)), abs=1e-15)
    assert ol.silu(50.0) == pytest.approx(50.0, abs=1e-15)
    assert abs(ol.silu(-50.0)) < 1e-19 and np.isfinite(ol.silu(-1000.0))
    # its only minimum: g = -W(1/e) - 1 ~ -1.27846, value ~ -0.27846
    g = np.linspace(-3, 0, 300001)
    i = int(np.argmin(ol.silu(g)))
    assert g[i] == pytest.approx(-1.27846, abs=1e-4)
    assert ol.silu(g[i]) == pytest.approx(-0.27846, abs=1e-4)


def test_gated_mlp_halves():
    rng = np.random.default_rng(3)
    x, wg, wu = rng.standard_normal((4, 6)), rng.standard_normal((5, 6)), rng.standard_normal((5, 6))
    got = ol.gated_mlp_up(x, np.concatenate([wg, wu]))
    g, u = np.array(loops(x, wg)), np.array(loops(x, wu))
    np.testing.assert_allclose(got, g / (1.0 + np.exp(-g)) * u, rtol=0, atol=1e-12)


def test_residual_adds():
    rng = np.random.default_rng(4)
    y, x, w = rng.standard_normal((3, 5)), rng.standard_normal((3, 4)), rng.standard_normal((5, 4))
    np.testing.assert_allclose(ol.residual(y, x, w), y + np.array(loops(x, w)), rtol=0, atol=1e-12)


def test_bf16_inputs_are_decoded_exactly():
    bits = np.array([[0x3F80, 0x4000], [0xBF80, 0x3F00]], np.uint16)   # 1, 2 / -1, 0.5
    w = np.array([[0x3F80, 0x3F80]], np.uint16)                         # 1, 1
    np.testing.assert_array_equal(ol.linear(bits, w), [[3.0], [-0.5]])


def test_pin_catches_transposed_weight(monkeypatch):
    rng = np.random.default_rng(5)
    x, w = rng.standard_normal((4, 4)), rng.standard_normal((4, 4))
    ref = np.array(loops(x, w))
    monkeypatch.setattr(ol, "linear", lambda a, b: np.asarray(a) @ np.asarray(b))
    assert not np.allclose(ol.linear(x, w), ref)


def test_pin_catches_swapped_gate_and_up():
    rng = np.random.default_rng(6)
    x, wg, wu = rng.standard_normal((4, 6)), rng.standard_normal((5, 6)), rng.standard_normal((5, 6))
    right = ol.gated_mlp_up(x, np.concatenate([wg, wu]))
    swapped = ol.gated_mlp_up(x, np.concatenate([wu, wg]))
    assert not np.allclose(right, swapped)
