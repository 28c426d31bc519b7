"""Pins for the oracle's LM head and log-sum-exp (CPU): a one-hot hidden row
selects one column of W, a constant W gives c * sum(h) + ln V, and tiny
products equal explicit sums."""
import math

import numpy as np

from oracle import lmhead as olm
from oracle import select as osel


def test_one_hot_row_picks_a_weight_column():
    rng = np.random.default_rng(0)
    V, H = 50, 16
    W = rng.normal(size=(V, H))
    h = np.zeros((3, H))
    h[0, 5] = 1.0
    h[1, 0] = 1.0
    h[2, 15] = 1.0
    lse, lg = olm.lse_rows(h, W)
    for r, j in enumerate((5, 0, 15)):
        assert np.array_equal(lg[r], W[:, j])
        m = W[:, j].max()
        assert abs(lse[r] - (m + math.log(np.exp(W[:, j] - m).sum()))) < 1e-12


def test_constant_weight_closed_form():
    rng = np.random.default_rng(1)
    V, H, c = 1000, 32, 0.25
    h = rng.normal(size=(4, H))
    lse, _ = olm.lse_rows(h, np.full((V, H), c))
    assert np.abs(lse - (c * h.sum(axis=1) + math.log(V))).max() < 1e-12


def test_tiny_products_equal_explicit_sums():
    rng = np.random.default_rng(2)
    h = rng.normal(size=(3, 5))
    W = rng.normal(size=(7, 5))
    lg = olm.logits64(h, W, rows=[2, 0])
    for i, r in enumerate((2, 0)):
        for v in range(7):
            assert abs(lg[i, v] - sum(h[r, k] * W[v, k] for k in range(5))) < 1e-12
    lse, _ = olm.lse_rows(h, W)
    assert abs(lse[1] - osel.lse64(h[1] @ W.T)) == 0.0
