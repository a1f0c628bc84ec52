"""Pins for the oracle's EPIKV score (hidden-state change, causal rolling z-score, two bands).

A hand-worked fixture, closed forms (constant velocity, a linearly growing signal), the L2 norm
against numpy's, invariances (shift, scale, band swap) and Samuelson's bound on a z-score. No GPU.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def test_epikv_handworked():
    case = json.load(open(os.path.join(GOLDEN, "epikv_handworked.json")))
    hA = _f32(case["hA"])[None]
    hB = _f32(case["hB"])[None]
    g, sc = O.epikv_score(hA, hB, case["window"], case["eps"], "f32")
    np.testing.assert_allclose(g[0, 0], case["gA"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g[1, 0], case["gB"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sc[0], case["score"], rtol=1e-12, atol=1e-12)


def test_signal_is_the_l2_norm_of_the_step():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((3, 40, 24)).astype(np.float32)
    g, _ = O.epikv_score(h, h, 8, 1e-6, "f32")
    want = np.linalg.norm(h[:, 1:].astype(np.float64) - h[:, :-1].astype(np.float64), axis=-1)
    np.testing.assert_allclose(g[0, :, 1:], want, rtol=1e-12)
    assert (g[:, :, 0] == 0).all()


def test_bf16_inputs_are_widened_exactly():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 30, 16))
    bits = O.f64_to_bf16_bits(x)
    vals = O.bf16_bits_to_f64(bits).astype(np.float32)
    gb, sb = O.epikv_score(bits, bits[::-1].copy(), 5, 1e-3, "bf16")
    gf, sf = O.epikv_score(vals, vals[::-1].copy(), 5, 1e-3, "f32")
    np.testing.assert_array_equal(gb, gf)
    np.testing.assert_array_equal(sb, sf)


def test_constant_velocity_gives_zero():
    """h(t) = h0 + t v: the step is the same every token, so every window has sigma 0 and z = 0."""
    t = np.arange(64, dtype=np.float32)[:, None]
    h = _f32(np.array([1.0, -2.0, 0.5]) + t * np.array([0.25, 0.5, -1.0]))[None]
    _, sc = O.epikv_score(h, h * 3, 16, 1e-3, "f32")
    assert np.abs(sc).max() < 1e-9  # zero up to the rounding of a mean of equal fp64 values


@pytest.mark.parametrize("W", [2, 5, 16])
def test_linear_signal_closed_form(W):
    """g(t) = a t: over a full window the values are a(t-W+1) .. a t, so mu = a(t - (W-1)/2) and
    sigma = a sqrt((W^2 - 1)/12), and z = sqrt(3 (W - 1)/(W + 1)) as eps -> 0. Layer B moves at a
    constant speed (its windows have sigma 0 and g = mu exactly, so z_B = 0 for any eps > 0), so the
    score is z_A; eps = 1e-300 stands for the limit."""
    a, N = 0.5, 48
    c = np.concatenate([[0.0], np.cumsum(a * np.arange(1, N))])  # c(t) - c(t-1) = a t
    hA = _f32(np.stack([c, np.zeros(N)], axis=1))[None]
    hB = _f32(np.stack([np.arange(N, dtype=np.float64), np.zeros(N)], axis=1))[None]
    g, sc = O.epikv_score(hA, hB, W, 1e-300, "f32")
    np.testing.assert_allclose(g[0, 0, 1:], a * np.arange(1, N), rtol=1e-6)
    want = math.sqrt(3.0 * (W - 1) / (W + 1))
    np.testing.assert_allclose(sc[0, W:], want, rtol=1e-5)


def test_invariances():
    rng = np.random.default_rng(3)
    hA = rng.standard_normal((2, 80, 32)).astype(np.float32)
    hB = rng.standard_normal((2, 80, 32)).astype(np.float32)
    _, s = O.epikv_score(hA, hB, 12, 0.0, "f32")
    # a band swap negates the score
    _, s_sw = O.epikv_score(hB, hA, 12, 0.0, "f32")
    np.testing.assert_allclose(s_sw, -s, rtol=0, atol=1e-12)
    # a constant added to every token of a layer changes no step
    _, s_sh = O.epikv_score(hA + np.float32(3.0), hB, 12, 0.0, "f32")
    np.testing.assert_allclose(s_sh, s, rtol=1e-6, atol=1e-6)
    # scaling a layer by a power of two scales its g exactly, and the z-score not at all
    _, s_sc = O.epikv_score(hA * np.float32(8.0), hB * np.float32(0.25), 12, 0.0, "f32")
    np.testing.assert_allclose(s_sc, s, rtol=1e-12, atol=1e-12)


def test_samuelson_bound():
    """A value lies within sqrt(n - 1) population standard deviations of the mean of any n values
    containing it, so |z| <= sqrt(min(t, W) - 1) as eps -> 0 (a sample std would allow more). Layer B
    moves at a constant speed (z_B = 0); eps = 1e-300 stands for the limit."""
    rng = np.random.default_rng(4)
    h = np.cumsum(rng.standard_normal((1, 200, 8)) * rng.gamma(0.5, 1.0, (1, 200, 1)), axis=1).astype(np.float32)
    flat = np.zeros_like(h)
    flat[..., 0] = np.arange(200, dtype=np.float32)
    for W in (3, 10, 50):
        _, sc = O.epikv_score(h, flat, W, 1e-300, "f32")
        n = np.minimum(np.arange(200), W)
        bound = np.sqrt(np.maximum(n - 1, 0)) + 1e-9
        assert (np.abs(sc[0]) <= bound).all()
    # the bound is reached: one jump after a flat stretch
    h2 = np.zeros((1, 30, 2), np.float32)
    h2[0, :, 0] = np.arange(30)
    h2[0, 20:, 0] += 10.0  # g = 1 everywhere except 11 at t = 20
    flat2 = np.zeros_like(h2)
    flat2[0, :, 0] = np.arange(30)
    _, sc = O.epikv_score(h2, flat2, 10, 1e-300, "f32")
    np.testing.assert_allclose(sc[0, 20], 3.0, rtol=1e-12)  # n = 10: sqrt(9)
