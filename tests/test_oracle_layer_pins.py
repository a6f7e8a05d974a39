"""Pins of the oracle's MLP half of a decoder layer and of its head
(``oracle.spark_layer``) against facts other than the oracle itself: the
standard normal CDF's table values, limits, brute force written as plain
Python loops on tiny inputs, and special cases with a known result.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import OracleGeometry

# Phi(z), the standard normal CDF, as printed in the usual tables (to 16
# digits): Phi(1) - Phi(-1) = 0.6826894921370859 is the "one sigma" mass.
PHI_TABLE = {
    -2.0: 0.022750131948179195,
    -1.0: 0.15865525393145707,
    1.0: 0.8413447460685429,
    2.0: 0.9772498680518208,
}


def test_gelu_is_x_times_the_normal_cdf():
    for z, phi in PHI_TABLE.items():
        assert oracle.gelu_erf(np.array([z]))[0] == pytest.approx(z * phi, rel=1e-14, abs=0)


def test_gelu_zero_and_limits():
    assert oracle.gelu_erf(np.array([0.0]))[0] == 0.0
    big = np.array([10.0, 40.0])
    np.testing.assert_allclose(oracle.gelu_erf(big), big, rtol=1e-15)
    np.testing.assert_allclose(oracle.gelu_erf(-big), 0.0, atol=1e-20)


def test_gelu_is_the_erf_form_not_the_tanh_approximation():
    z = 1.0
    tanh_form = 0.5 * z * (1 + math.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))
    exact = z * PHI_TABLE[1.0]
    assert abs(tanh_form - exact) > 1e-4          # the two differ visibly at z = 1
    assert abs(oracle.gelu_erf(np.array([z]))[0] - exact) < 1e-14


def _tiny_mlp_weights(rng, hidden, inter):
    return {
        "norm_w": (1 + 0.1 * rng.standard_normal(hidden)).astype(np.float32),
        "gate_w": (rng.standard_normal((inter, hidden)) / math.sqrt(hidden)).astype(np.float32),
        "up_w": (rng.standard_normal((inter, hidden)) / math.sqrt(hidden)).astype(np.float32),
        "down_w": (rng.standard_normal((hidden, inter)) / math.sqrt(inter)).astype(np.float32),
    }


def _loop_mlp(h, w, eps):
    """The MLP half of a layer as plain loops over Python floats."""
    hidden = len(h)
    inter = len(w["gate_w"])
    ss = sum(float(v) * float(v) for v in h)
    inv = 1.0 / math.sqrt(ss / hidden + eps)
    x = [float(h[c]) * inv * float(w["norm_w"][c]) for c in range(hidden)]
    m = []
    for j in range(inter):
        g = sum(float(w["gate_w"][j][c]) * x[c] for c in range(hidden))
        u = sum(float(w["up_w"][j][c]) * x[c] for c in range(hidden))
        m.append(0.5 * g * (1 + math.erf(g / math.sqrt(2))) * u)
    return [float(h[r]) + sum(float(w["down_w"][r][j]) * m[j] for j in range(inter))
            for r in range(hidden)]


def test_mlp_matches_plain_loops():
    rng = np.random.default_rng(7)
    geom = OracleGeometry(hidden=24)
    w = _tiny_mlp_weights(rng, 24, 40)
    h = rng.standard_normal((3, 24)).astype(np.float32)
    got = oracle.mlp_block(geom, h, w)["out"]
    for b in range(3):
        np.testing.assert_allclose(got[b], _loop_mlp(h[b], w, geom.eps), rtol=1e-12, atol=1e-12)


def test_mlp_with_zero_down_returns_h_exactly():
    rng = np.random.default_rng(8)
    geom = OracleGeometry(hidden=16)
    w = _tiny_mlp_weights(rng, 16, 32)
    w["down_w"] = np.zeros_like(w["down_w"])
    h = rng.standard_normal((2, 16)).astype(np.float32)
    np.testing.assert_array_equal(oracle.mlp_block(geom, h, w)["out"], h.astype(np.float64))


def test_mlp_gate_and_up_are_not_interchangeable():
    # x = rms(h) * w with h = 1 and w = 1 is the all-ones vector.  Gate row 0
    # sums to -10 (GELU ~ -7.7e-23), up row 0 sums to +5: the product is ~0.
    # Swapped, it would be gelu(5) * -10 = -50.
    geom = OracleGeometry(hidden=8, eps=0.0)
    w = {
        "norm_w": np.ones(8, np.float32),
        "gate_w": np.full((1, 8), -10.0 / 8, np.float32),
        "up_w": np.full((1, 8), 5.0 / 8, np.float32),
        "down_w": np.ones((8, 1), np.float32),
    }
    h = np.ones((1, 8), np.float32)
    r = oracle.mlp_block(geom, h, w)
    np.testing.assert_allclose(r["x"][0], 1.0, rtol=1e-15)
    assert abs(r["m"][0][0]) < 1e-20
    np.testing.assert_allclose(r["out"][0], 1.0, atol=1e-20)


def test_head_logits_match_plain_loops_and_one_hot_rows():
    rng = np.random.default_rng(9)
    geom = OracleGeometry(hidden=12)
    norm_w = (1 + 0.1 * rng.standard_normal(12)).astype(np.float32)
    embed = rng.standard_normal((30, 12)).astype(np.float32)
    h = rng.standard_normal((2, 12)).astype(np.float32)
    got = oracle.head_logits(geom, h, norm_w, embed)
    for b in range(2):
        inv = 1.0 / math.sqrt(sum(float(v) ** 2 for v in h[b]) / 12 + geom.eps)
        x = [float(h[b][c]) * inv * float(norm_w[c]) for c in range(12)]
        want = [sum(float(embed[v][c]) * x[c] for c in range(12)) for v in range(30)]
        np.testing.assert_allclose(got[b], want, rtol=1e-12, atol=1e-12)
    # one-hot rows: logit v is component v of the normed hidden state
    onehot = np.eye(12, dtype=np.float32)
    x0 = oracle.rms_norm(h[0], norm_w, geom.eps)
    np.testing.assert_allclose(oracle.head_logits(geom, h[:1], norm_w, onehot)[0], x0, rtol=1e-15)
