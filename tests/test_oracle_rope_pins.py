"""Pins of the float64 rotary / YaRN / bias oracle against things other than
its own formulas.

A plausible mistake -- pairing dims (2i, 2i+1) instead of (i, i + D/2), a
sign flip in the rotation, frequencies in the wrong order, the YaRN ramp
reversed or applied to the wrong end, the temperature on the logits twice or
not at all, the bias added after the rotation -- fails at least one test.
Source of the definitions: the rotary encoding of RoFormer and the YaRN
paper's NTK-by-parts interpolation and temperature, which the model overview
of "GPT-OSS on day 0" names.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(300)


def _inv_freq(D=64, base=10000.0):
    return oracle.yarn_inv_freq(D, base, 1.0, 4096, 32.0, 1.0)[0]


def test_position_zero_is_identity_times_factor():
    x = RNG.normal(size=(3, 4, 64))
    f = RNG.uniform(0, 2, size=32)
    np.testing.assert_allclose(oracle.rope(x, [0, 0, 0], f, 1.7), 1.7 * x, rtol=0, atol=1e-15)


def test_rotation_preserves_norms_per_plane():
    x = RNG.normal(size=(50, 3, 64))
    pos = RNG.integers(0, 200000, size=50)
    f = _inv_freq()
    y = oracle.rope(x, pos, f)
    plane = lambda z: z[..., :32] ** 2 + z[..., 32:] ** 2  # noqa: E731
    np.testing.assert_allclose(plane(y), plane(x), rtol=1e-12, atol=1e-12)


def test_one_hot_rotates_in_its_plane():
    # e_i at position p -> cos(p f_i) e_i + sin(p f_i) e_{i+D/2}; e_{i+D/2} -> -sin e_i + cos e_{i+D/2}
    D, p = 8, 3
    f = np.array([1.0, 0.5, 0.25, 0.125])
    for i in range(4):
        e = np.zeros((1, 1, D))
        e[0, 0, i] = 1.0
        y = oracle.rope(e, [p], f)[0, 0]
        want = np.zeros(D)
        want[i], want[i + 4] = math.cos(p * f[i]), math.sin(p * f[i])
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-15)
        e = np.zeros((1, 1, D))
        e[0, 0, i + 4] = 1.0
        y = oracle.rope(e, [p], f)[0, 0]
        want = np.zeros(D)
        want[i], want[i + 4] = -math.sin(p * f[i]), math.cos(p * f[i])
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-15)


def test_dot_products_depend_only_on_relative_position():
    q = RNG.normal(size=(1, 1, 64))
    k = RNG.normal(size=(1, 1, 64))
    f = _inv_freq()
    def dot(m, n):
        return float((oracle.rope(q, [m], f) * oracle.rope(k, [n], f)).sum())
    for m, n in [(5, 2), (1000, 17), (70000, 69999)]:
        for shift in (1, 123, 40000):
            assert abs(dot(m + shift, n + shift) - dot(m, n)) < 1e-9


def test_rotations_compose():
    x = RNG.normal(size=(4, 2, 16))
    f = RNG.uniform(0, 1, size=8)
    a, b = np.array([1, 7, 100, 3000]), np.array([2, 0, 55, 9])
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, f), b, f), oracle.rope(x, a + b, f),
                               rtol=0, atol=1e-11)


def test_plain_rope_frequencies_decrease_geometrically():
    f = _inv_freq(64, 150000.0)
    assert f[0] == 1.0
    np.testing.assert_allclose(f[1:] / f[:-1], 150000.0 ** (-2 / 64), rtol=1e-14)
    assert oracle.yarn_inv_freq(64, 150000.0, 1.0, 4096, 32.0, 1.0)[1] == 1.0


def test_yarn_keeps_high_frequencies_and_divides_low_ones():
    D, base, s, L0, bf, bs = 64, 150000.0, 32.0, 4096, 32.0, 1.0
    plain = _inv_freq(D, base)
    yarn, mscale = oracle.yarn_inv_freq(D, base, s, L0, bf, bs)
    turns = L0 * plain / (2 * math.pi)  # rotations of each plane over the original context
    fast, slow = turns > bf, turns < bs
    assert fast.any() and slow.any() and (~fast & ~slow).any()
    np.testing.assert_array_equal(yarn[fast], plain[fast])          # many turns: unchanged
    np.testing.assert_allclose(yarn[slow], plain[slow] / s, rtol=1e-15)  # < 1 turn: interpolated
    mid = ~fast & ~slow
    assert np.all(yarn[mid] < plain[mid]) and np.all(yarn[mid] > plain[mid] / s)
    assert abs(mscale - (0.1 * math.log(32.0) + 1.0)) < 1e-15


def test_yarn_ramp_midpoint():
    # choose the original context so that plane j turns exactly (alpha + beta) / 2 times:
    # there the ramp is 1/2 and the frequency the mean of theta and theta / s
    D, base, s, alpha, beta, j = 64, 10000.0, 8.0, 2.0, 10.0, 9
    theta_j = base ** (-2.0 * j / D)
    L0 = (alpha + beta) / 2 * 2 * math.pi / theta_j
    yarn, _ = oracle.yarn_inv_freq(D, base, s, L0, beta, alpha)
    np.testing.assert_allclose(yarn[j], theta_j * (1 + 1 / s) / 2, rtol=1e-12)


def test_bias_is_added_before_the_rotation():
    # rope is linear: rope(x + b) = rope(x) + rope(b); adding b after the rotation differs
    T, H, D = 5, 2, 16
    q, k, v = RNG.normal(size=(T, H, D)), RNG.normal(size=(T, 1, D)), RNG.normal(size=(T, 1, D))
    bq, bk, bv = RNG.normal(size=(H, D)), RNG.normal(size=(1, D)), RNG.normal(size=(1, D))
    pos = np.array([0, 1, 9, 100, 5000])
    f = RNG.uniform(0, 1, size=D // 2)
    q2, k2, v2 = oracle.qkv_bias_rope(q, k, v, bq, bk, bv, pos, f, 1.3)
    bq_t = np.broadcast_to(bq, q.shape)
    np.testing.assert_allclose(q2, oracle.rope(q, pos, f, 1.3) + oracle.rope(bq_t, pos, f, 1.3), atol=1e-13)
    assert np.abs(q2 - (oracle.rope(q, pos, f, 1.3) + 1.3 * bq_t)).max() > 1e-2
    np.testing.assert_allclose(v2, v + bv, atol=0)
    q0, k0, v0 = oracle.qkv_bias_rope(q, k, v, None, None, None, pos, f, 1.0)
    np.testing.assert_allclose(q0, oracle.rope(q, pos, f), atol=0)
    np.testing.assert_array_equal(v0, v)
