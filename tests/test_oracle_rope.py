"""Pins of the rotary-embedding oracle against facts that do not depend on it:
closed forms of single channels, the identity at position 0, orthogonality
(pair norms kept, inverse undoes forward) and the relative-position property
that makes RoPE useful: <R_m q, R_n k> depends only on m - n."""
import math

import numpy as np
import pytest

from oracle import rope as R


def test_position_zero_is_identity():
    x = np.random.default_rng(0).standard_normal((3, 2, 64))
    assert np.array_equal(R.rope(x, [0, 0, 0]), x)


def test_first_pair_closed_form():
    # theta_0 = base^0 = 1: channel 0 rotates with channel d/2 by exactly p radians
    d, p = 128, 77
    x = np.zeros((1, 1, d))
    x[0, 0, 0], x[0, 0, d // 2] = 0.25, -1.5
    y = R.rope(x, [p])
    assert y[0, 0, 0] == pytest.approx(0.25 * math.cos(p) + 1.5 * math.sin(p), abs=1e-14)
    assert y[0, 0, d // 2] == pytest.approx(-1.5 * math.cos(p) + 0.25 * math.sin(p), abs=1e-14)


def test_last_pair_frequency():
    # theta_{d/2-1} = base^(-(d-2)/d); with base 10000, d = 4 that is 10000^-0.5 = 0.01
    x = np.array([[[0.0, 1.0, 0.0, 0.0]]])     # channel 1 pairs with channel 3
    y = R.rope(x, [50])
    assert y[0, 0, 1] == pytest.approx(math.cos(0.5), abs=1e-14)
    assert y[0, 0, 3] == pytest.approx(math.sin(0.5), abs=1e-14)


def test_pair_norms_kept_and_inverse_undoes_forward():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 3, 128))
    p = rng.integers(0, 200000, size=50)
    y = R.rope(x, p)
    n_x = x[..., :64] ** 2 + x[..., 64:] ** 2
    n_y = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(n_x, n_y, rtol=1e-12, atol=1e-12)
    assert np.allclose(R.rope(y, p, inverse=True), x, rtol=0, atol=1e-9)


def test_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    ref = float(np.sum(R.rope(q, [9]) * k))               # m - n = 9 with n = 0
    for m in (9, 100, 4096 + 9, 65000):
        s = float(np.sum(R.rope(q, [m]) * R.rope(k, [m - 9])))
        assert s == pytest.approx(ref, abs=1e-8)
