"""Pins of the oracle's rotary position embedding (``oracle.rope``).

The pages name RoPE among the model's techniques without a formula; the
oracle takes the original rotary embedding on pairs (2i, 2i+1) with
theta_i = base^(-2i/d).  These tests pin it to facts that do not come from
the oracle:
- the rotation of a unit vector by a whole number of radians: textbook
  values of cos 1, sin 1, cos 2, sin 2;
- the frequency exponent: with base 10^4 and d = 4 the second pair turns by
  n / 100 (a wrong exponent gives another angle);
- invariants: position 0 is the identity, every pair keeps its length, the
  inverse undoes the rotation, and dot products depend only on the position
  difference (the property rotary embeddings are built for);
- the gradient of attention on rotated Q and K, with the inverse rotation
  applied to dQ and dK, against central finite differences with the pages'
  epsilon 1e-5 and relative-error threshold 1e-4.
"""
import math

import numpy as np
import pytest

import oracle

rng = np.random.default_rng(4321)

COS1, SIN1 = 0.5403023058681398, 0.8414709848078965
COS2, SIN2 = -0.4161468365471424, 0.9092974268256817


def test_unit_vector_turns_by_position_radians():
    # d = 2: theta_0 = 1 for any base; rows at positions 0, 1, 2
    x = np.array([[1.0, 0.0], [1.0, 0.0], [1.0, 0.0]])
    y = oracle.rope(x, base=10000.0)
    np.testing.assert_allclose(y, [[1.0, 0.0], [COS1, SIN1], [COS2, SIN2]], rtol=0, atol=1e-15)
    x2 = np.array([[0.0, 1.0], [0.0, 1.0]])
    y2 = oracle.rope(x2)
    np.testing.assert_allclose(y2[1], [-SIN1, COS1], rtol=0, atol=1e-15)


def test_frequency_exponent():
    # d = 4, base 1e4: theta_1 = 1e4^(-2/4) = 1/100; at position 100 the
    # second pair turns by exactly 1 radian, the first by 100 radians
    N, d = 101, 4
    x = np.zeros((N, d))
    x[:, 2] = 1.0
    y = oracle.rope(x, base=10000.0)
    np.testing.assert_allclose(y[100, 2:], [COS1, SIN1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(y[100, :2], [0.0, 0.0], atol=0)


def test_position_zero_is_identity_and_lengths_kept():
    x = rng.standard_normal((3, 37, 16))
    y = oracle.rope(x, base=500.0)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])
    nx = np.hypot(x[..., 0::2], x[..., 1::2])
    ny = np.hypot(y[..., 0::2], y[..., 1::2])
    np.testing.assert_allclose(ny, nx, rtol=1e-13, atol=0)


def test_inverse_undoes_rotation():
    x = rng.standard_normal((2, 5, 64, 8))
    back = oracle.rope(oracle.rope(x), inverse=True)
    np.testing.assert_allclose(back, x, rtol=0, atol=1e-12)
    assert np.abs(oracle.rope(x) - x).max() > 0.1


def test_dot_depends_on_position_difference_only():
    d, N = 16, 40
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    Q = oracle.rope(np.tile(q, (N, 1)))
    K = oracle.rope(np.tile(k, (N, 1)))
    for m, n in ((5, 2), (17, 3), (30, 30)):
        for s in (1, 7):
            a = Q[m] @ K[n]
            b = Q[m + s] @ K[n + s]
            assert abs(a - b) <= 1e-12 * max(1.0, abs(a))


def _loss(q, k, v, do, s):
    o, _ = oracle.attn_fwd(oracle.rope(q), oracle.rope(k), v, s, True)
    return float((o * do).sum())


def test_rotated_attention_gradient_by_finite_differences():
    B, H, Hkv, N, d = 1, 2, 1, 12, 8
    q, k = rng.standard_normal((B, H, N, d)), rng.standard_normal((B, Hkv, N, d))
    v, do = rng.standard_normal((B, Hkv, N, d)), rng.standard_normal((B, H, N, d))
    s = 1 / math.sqrt(d)
    dqr, dkr, _ = oracle.attn_bwd(oracle.rope(q), oracle.rope(k), v, do, s, True)
    grads = {"q": oracle.rope(dqr, inverse=True), "k": oracle.rope(dkr, inverse=True)}
    eps, tol = 1e-5, 1e-4
    for name, a in (("q", q), ("k", k)):
        for idx in np.ndindex(a.shape):
            orig = a[idx]
            a[idx] = orig + eps
            lp = _loss(q, k, v, do, s)
            a[idx] = orig - eps
            lm = _loss(q, k, v, do, s)
            a[idx] = orig
            fd = (lp - lm) / (2 * eps)
            an = grads[name][idx]
            assert abs(fd - an) / max(abs(fd), abs(an), 1e-6) < tol, (name, idx, fd, an)


def test_rejects_odd_width():
    with pytest.raises(ValueError):
        oracle.rope(np.zeros((4, 3)))
