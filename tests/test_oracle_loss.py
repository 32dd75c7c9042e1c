"""Pins of the masked-loss oracle: closed forms of the cross-entropy, the
ignore rule, the gradient's row sums and the page's statement that the
token-weighted reduction over sequence-parallel ranks gives every rank the
loss of the whole sequence."""
import math

import numpy as np
import pytest

from oracle import loss as L


def test_uniform_logits_give_log_vocab():
    V = 50000
    s, n, mean = L.masked_loss(np.full((3, V), 1.25), [7, 0, V - 1])
    assert n == 3 and mean == pytest.approx(math.log(V), abs=1e-12)


def test_two_class_closed_form():
    # logits (a, b), label 0: loss = log(1 + e^(b - a))
    a, b = 2.0, -0.5
    assert L.token_losses([[a, b]], [0])[0] == pytest.approx(math.log1p(math.exp(b - a)), abs=1e-15)


def test_ignored_tokens_count_for_nothing():
    x = np.random.default_rng(0).standard_normal((5, 11))
    s, n, mean = L.masked_loss(x, [-100] * 5)
    assert (s, n, mean) == (0.0, 0, 0.0)
    full = L.masked_loss(x, [1, -100, 3, -100, 4])
    part = L.masked_loss(x[[0, 2, 4]], [1, 3, 4])
    assert full[1] == 3 and full[0] == pytest.approx(part[0], abs=1e-12)


def test_gradient_rows_sum_to_zero_and_match_finite_differences():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 7))
    g = L.logits_grad(x, [3, -100], 0.5)
    assert np.allclose(g.sum(axis=1), 0.0, atol=1e-15) and not g[1].any()
    eps = 1e-6
    for j in range(7):
        xp, xm = x.copy(), x.copy()
        xp[0, j] += eps
        xm[0, j] -= eps
        fd = (L.token_losses(xp, [3, -100])[0] - L.token_losses(xm, [3, -100])[0]) / (2 * eps) * 0.5
        assert g[0, j] == pytest.approx(fd, abs=1e-8)


def test_sequence_parallel_reduction_gives_the_whole_sequence_loss():
    rng = np.random.default_rng(2)
    T, V, sp = 64, 30, 4
    x = rng.standard_normal((T, V)) * 3
    lab = rng.integers(0, V, size=T)
    lab[rng.random(T) < 0.3] = -100
    whole = L.masked_loss(x, lab)[2]
    c = T // sp
    parts = [L.masked_loss(x[r * c:(r + 1) * c], lab[r * c:(r + 1) * c]) for r in range(sp)]
    red = L.reduce_sequence_parallel_loss([p[2] for p in parts], [p[1] for p in parts])
    assert red == pytest.approx(whole, abs=1e-12)
