"""Pins of the oracle's ffn_norm (RMSNorm: h * w / sqrt(mean(h^2) + eps), the
fused add+RMSNorm kernel on "ferrox-cuda 0.14.0 — src/gpu.rs" applied to the
hidden state as moe_layer on "aprender-serve 0.70.2 —
forward_qwen3_moe_resident.rs" does).  Each test fixes a value the
definition determines without re-evaluating the formula: closed forms for
constant and one-hot inputs, invariances, and degenerate cases."""
import numpy as np
import pytest


def test_constant_vector_closed_form(orc):
    # h = c everywhere: mean(h^2) = c^2, so out = c * w / sqrt(c^2 + eps)
    n, c, eps = 64, 3.0, 0.25
    w = np.linspace(0.5, 2.0, n).astype(np.float32)
    got = orc.rmsnorm(np.full(n, c, np.float32), w, eps)
    np.testing.assert_allclose(got, 3.0 * w.astype(np.float64) / np.sqrt(9.25), rtol=1e-15)


def test_one_hot_closed_form(orc):
    # h = v at index k only: mean(h^2) = v^2 / n; with eps = 0 the output is
    # sign(v) * sqrt(n) * w_k at k and 0 elsewhere
    n, k, v = 256, 37, -0.75
    h = np.zeros(n, np.float32)
    h[k] = v
    w = (1.0 + np.arange(n) / n).astype(np.float32)
    got = orc.rmsnorm(h, w, 0.0)
    want = np.zeros(n)
    want[k] = -np.sqrt(n) * float(w[k])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=0)


def test_unit_rms_and_scale_invariance(orc):
    g = np.random.default_rng(5)
    h = g.standard_normal(512).astype(np.float32)
    ones = np.ones(512, np.float32)
    out = orc.rmsnorm(h, ones, 0.0)
    assert np.mean(out ** 2) == pytest.approx(1.0, rel=1e-12)
    # positive scaling of h leaves the output unchanged (eps = 0); negation negates it
    np.testing.assert_allclose(orc.rmsnorm(4.0 * h, ones, 0.0), out, rtol=1e-12)
    np.testing.assert_allclose(orc.rmsnorm(-h, ones, 0.0), -out, rtol=1e-12)


def test_linear_in_weight(orc):
    g = np.random.default_rng(6)
    h = g.standard_normal(128).astype(np.float32)
    w1 = g.standard_normal(128).astype(np.float32)
    w2 = g.standard_normal(128).astype(np.float32)
    a = orc.rmsnorm(h, w1, 1e-5) + orc.rmsnorm(h, w2, 1e-5)
    b = orc.rmsnorm(h, (w1.astype(np.float64) + w2).astype(np.float32), 1e-5)
    # w1 + w2 is rounded to f32 once: compare within that rounding
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)


def test_zero_input_stays_zero(orc):
    out = orc.rmsnorm(np.zeros(32, np.float32), np.ones(32, np.float32), 1e-6)
    assert np.all(out == 0.0)


def test_rows_are_normed_independently(orc):
    g = np.random.default_rng(7)
    H = g.standard_normal((3, 64)).astype(np.float32)
    w = np.ones(64, np.float32)
    both = orc.rmsnorm(H, w, 1e-5)
    for t in range(3):
        np.testing.assert_array_equal(both[t], orc.rmsnorm(H[t], w, 1e-5))
