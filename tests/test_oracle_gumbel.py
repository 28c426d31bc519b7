"""Pins for the oracle's Gumbel top-k (temperature > 0) and its noise (CPU).

What fixes them independently of the oracle's code: the published
known-answer vectors of Philox4x32-10 (Salmon et al., SC 2011, as shipped
with the Random123 library), the natural logarithm itself, the Gumbel(0, 1)
distribution's mean (Euler's constant), variance (pi^2 / 6) and CDF
exp(-exp(-x)), the Gumbel-max property (the argmax of logit / tau + g is a
draw from softmax(logit / tau)), the temperature -> 0 limit (deterministic
top-k), and brute-force enumeration of the whole beam x vocab grid.
"""
import math

import numpy as np
import pytest
import scipy.stats

import synth
from oracle import gumbel as G
from oracle import select as osel
from oracle import trie as otrie

F32 = np.float32


@pytest.mark.parametrize("ctr,key,want", [
    ((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
    ((0xffffffff,) * 4, (0xffffffff,) * 2, (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
    ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
     (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1)),
])
def test_philox_known_answers(ctr, key, want):
    out = G.philox4x32_10(*[np.uint32(c) for c in ctr], *key)
    assert tuple(int(o) for o in out) == want


def test_ln_matches_natural_log():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(2.0 ** -25, 1, 50000), rng.uniform(1, 20, 50000),
                        [2.0 ** -25, 1 - 2.0 ** -24, 1.0, 2.0, 0.5, math.sqrt(2), math.e, 17.328]]).astype(F32)
    got = G.ln_f32(x).astype(np.float64)
    want = np.log(x.astype(np.float64))
    assert np.abs(got - want).max() < 1e-6
    assert G.ln_f32(np.array([1.0], F32))[0] == 0.0


def test_gumbel_distribution():
    g = G.gumbel(20261202, 0, 0, 0, np.arange(1_000_000)).astype(np.float64)
    n = len(g)
    assert abs(g.mean() - np.euler_gamma) < 5 * math.sqrt(math.pi ** 2 / 6 / n)
    assert abs(g.var() - math.pi ** 2 / 6) < 5 * (math.pi ** 2 / 6) * math.sqrt(4.4 / n)
    ks = scipy.stats.kstest(g, lambda x: np.exp(-np.exp(-x)))
    assert ks.statistic < 3e-3


def test_noise_depends_on_every_counter_field():
    base = G.gumbel(7, 1, 2, 3, np.array([4]))[0]
    for args in [(8, 1, 2, 3, 4), (7, 0, 2, 3, 4), (7, 1, 0, 3, 4), (7, 1, 2, 0, 4), (7, 1, 2, 3, 5),
                 (7 + (1 << 32), 1, 2, 3, 4)]:
        s, r, t, b, v = args
        assert G.gumbel(s, r, t, b, np.array([v]))[0] != base


def test_gumbel_max_draws_from_softmax():
    """One beam, W = K = 1, six open-vocabulary tokens: over many seeds the
    chosen token follows softmax(logit / tau)."""
    V, tau, n = 6, 0.7, 6000
    logits = np.array([[[0.5, -1.0, 1.5, 0.0, -0.3, 1.0]]], F32)
    counts = np.zeros(V)
    for seed in range(n):
        o = osel.beam_select(logits, np.zeros((1, 1), F32), np.zeros((1, 1), np.int64), np.array([1]),
                             np.full((1, 1, 1), -1, np.int32), None, None, 0, 0, 1, 1,
                             temperature=tau, seed=seed)
        counts[o["tokens"][0, 0]] += 1
    lp = logits[0, 0].astype(np.float64) / tau
    p = np.exp(lp - lp.max())
    p /= p.sum()
    assert scipy.stats.chisquare(counts, n * p).pvalue > 1e-4


def _tiny(seed, use_trie):
    wl = synth.WORKLOADS["tiny"]
    rng = np.random.default_rng(seed)
    items = synth.catalog(wl)
    trie = otrie.build_trie(items, wl.C) if use_trie else None
    W = 8
    logits = rng.normal(0, 2, size=(1, W, wl.V)).astype(F32)
    cum = np.sort(-np.abs(rng.normal(0, 3, size=(1, W))).astype(F32))[:, ::-1].copy()
    level = 1
    pre = items[rng.integers(0, len(items), size=W), :level]
    node = np.array([[trie.node_of_prefix(p) if trie else 0 for p in pre]])
    return wl, trie, logits, cum, node, level


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("use_trie", [True, False])
@pytest.mark.parametrize("K", [1, 3, 40])
def test_gumbel_two_stage_equals_bruteforce(seed, use_trie, K):
    wl, trie, logits, cum, node, level = _tiny(seed, use_trie)
    W = 8
    args = dict(temperature=0.8, seed=1000 + seed)
    o = osel.beam_select(logits, cum, node, np.array([W]), np.full((1, W, 3), -1, np.int32),
                         trie, wl.token_base(), level, level, W, K, **args)
    bf = osel.beam_select_bruteforce(logits, cum, node, np.array([W]), trie, wl.token_base(), level, W, K,
                                     step=level, **args)[0]
    n = o["n_live_out"][0]
    assert n == len(bf)
    assert o["tokens"][0, :n].tolist() == [x[0] for x in bf]
    assert o["parents"][0, :n].tolist() == [x[1] for x in bf]
    # the returned score is the noise-free cumulative log-probability
    assert o["cum_out"][0, :n].tolist() == [float(x[2]) for x in bf]
    for j in range(n):
        b, v = o["parents"][0, j], o["tokens"][0, j]
        lse = F32(osel.lse64(logits[0, b]))
        assert o["cum_out"][0, j] == F32(cum[0, b] + F32(logits[0, b, v] - lse))


def test_gumbel_changes_the_order():
    wl, trie, logits, cum, node, level = _tiny(0, False)
    W, K = 8, 8
    common = (logits, cum, node, np.array([W]), np.full((1, W, 3), -1, np.int32), trie, wl.token_base(),
              level, level, W, K)
    det = osel.beam_select(*common)
    noisy = osel.beam_select(*common, temperature=1.0, seed=5)
    assert det["tokens"][0].tolist() != noisy["tokens"][0].tolist()


@pytest.mark.parametrize("seed", range(3))
def test_small_temperature_is_deterministic_top_k(seed):
    wl, trie, logits, cum, node, level = _tiny(seed, True)
    W, K = 8, 5
    common = (logits, cum, node, np.array([W]), np.full((1, W, 3), -1, np.int32), trie, wl.token_base(),
              level, level, W, K)
    det = osel.beam_select(*common)
    cold = osel.beam_select(*common, temperature=1e-4, seed=seed)
    s = det["cum_out"][0].astype(np.float64)
    assert np.min(np.abs(np.diff(s))) > 1e-2    # these seeds have no near ties among the winners
    for k in ("tokens", "parents", "cum_out", "node_out", "n_live_out"):
        assert np.array_equal(det[k], cold[k])
