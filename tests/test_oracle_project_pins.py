"""Pins of the oracle's projections x -> k', q' ("Meccanismo Core" item 2: the projected key
and query whose halves are the sub-scores) against things other than its matmul:
  * one-hot features: x = e_d must return column d of the weights, placed by the stated
    layout (k' rows of w first, head-major, then half, then index; q' rows after them);
  * explicit loops over every index on tiny sizes;
  * linearity in x, and the magnitude sum against its definition on a sign-flipped input.
"""
import numpy as np

import oracle


def _w_row(H, S, which, h, half, s):
    return which * 2 * H * S + (h * 2 + half) * S + s


def test_one_hot_features_pick_weight_columns():
    B, T, D, H, S = 2, 3, 5, 3, 4
    rng = np.random.default_rng(0)
    w = rng.standard_normal((4 * H * S, D))
    for d in range(D):
        x = np.zeros((B, T, D))
        x[1, 2, d] = 1.0
        kp, qp, _ = oracle.project(x, w, H, S)
        assert kp.shape == (B, H, T, 2, S) and qp.shape == (B, H, T, 2, S)
        for h in range(H):
            for half in range(2):
                for s in range(S):
                    assert kp[1, h, 2, half, s] == w[_w_row(H, S, 0, h, half, s), d]
                    assert qp[1, h, 2, half, s] == w[_w_row(H, S, 1, h, half, s), d]
        # every other token is zero
        mask = np.ones((B, H, T), bool)
        mask[1, :, 2] = False
        assert not kp[mask].any() and not qp[mask].any()


def test_loops_on_tiny_sizes():
    B, T, D, H, S = 2, 2, 3, 2, 2
    rng = np.random.default_rng(1)
    x = rng.integers(-4, 5, (B, T, D)).astype(np.float64)
    w = rng.integers(-4, 5, (4 * H * S, D)).astype(np.float64)
    kp, qp, (mk, mq) = oracle.project(x, w, H, S)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                for half in range(2):
                    for s in range(S):
                        for which, out, mag in ((0, kp, mk), (1, qp, mq)):
                            n = _w_row(H, S, which, h, half, s)
                            acc = 0.0
                            am = 0.0
                            for d in range(D):
                                acc += x[b, t, d] * w[n, d]
                                am += abs(x[b, t, d] * w[n, d])
                            assert out[b, h, t, half, s] == acc   # small integers: exact
                            assert mag[b, h, t, half, s] == am


def test_linear_in_the_features():
    B, T, D, H, S = 1, 4, 16, 2, 3
    rng = np.random.default_rng(2)
    w = rng.integers(-8, 9, (4 * H * S, D)).astype(np.float64)
    x1 = rng.integers(-8, 9, (B, T, D)).astype(np.float64)
    x2 = rng.integers(-8, 9, (B, T, D)).astype(np.float64)
    k1, q1, _ = oracle.project(x1, w, H, S)
    k2, q2, _ = oracle.project(x2, w, H, S)
    k3, q3, _ = oracle.project(3 * x1 - x2, w, H, S)
    assert np.array_equal(k3, 3 * k1 - k2) and np.array_equal(q3, 3 * q1 - q2)
    # the magnitude ignores signs of the features
    _, _, (m1, n1) = oracle.project(x1, w, H, S)
    _, _, (m2, n2) = oracle.project(-x1, w, H, S)
    assert np.array_equal(m1, m2) and np.array_equal(n1, n2)
