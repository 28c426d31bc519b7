"""Pins for the oracle's beam expansion (CPU only).

Each pin is something the pages or plain mathematics fix independently of the
oracle's code: a hand-derived example, closed forms of log-sum-exp, exact
rational rounding of the score, brute-force enumeration of the whole
beam x vocab grid, and the invariants W=1 == greedy, top_k >= W == full pool,
illegal-item rate 0, and exhaustive catalog ranking.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import synth
from oracle import select as osel
from oracle import trie as otrie
from tests.golden import read_kv

F32 = np.float32


def _chain(wl, items, logit_fn, W=None, K=None, steps=None):
    """Run the oracle for ``steps`` decode steps; logit_fn(step, r, state) -> [R,W,V]."""
    W = W or wl.W
    K = K or wl.K
    T = wl.T if steps is None else steps
    trie = otrie.build_trie(items, wl.C) if wl.levels else None
    tb = wl.token_base()
    R = wl.R
    cum = np.zeros((R, W), F32)
    node = np.zeros((R, W), np.int64)
    n_live = np.ones(R, np.int32)
    slot = np.full((R, W, T), -1, np.int32)
    hist = [[[] for _ in range(W)] for _ in range(R)]
    outs = []
    for t in range(T):
        lg = logit_fn(t, hist, n_live)
        o = osel.beam_select(lg, cum, node, n_live, slot, trie, tb, t, t, W, K)
        outs.append(o)
        new_hist = [[[] for _ in range(W)] for _ in range(R)]
        for r in range(R):
            for j in range(o["n_live_out"][r]):
                new_hist[r][j] = hist[r][o["parents"][r, j]] + [int(o["tokens"][r, j])]
        hist = new_hist
        cum, node, n_live, slot = o["cum_out"], o["node_out"], o["n_live_out"], o["slot_out"]
    return outs, hist, trie


def test_golden_small_select():
    g = read_kv("select_small.txt")
    logits = np.log(np.array([g["probs0"], g["probs1"]], dtype=np.float64)).astype(F32)[None]
    cum = np.array([g["cum"]], dtype=F32)
    W, K = int(g["W"][0]), int(g["K"][0])
    cum_full = np.full((1, W), -np.inf, F32)
    cum_full[0, :2] = cum[0]
    o = osel.beam_select(logits, cum_full, np.zeros((1, W), np.int64), np.array([2]),
                         np.full((1, W, 1), -1, np.int32), None, None, 0, 0, W, K)
    assert o["tokens"][0].tolist() == [int(x) for x in g["tokens"]]
    assert o["parents"][0].tolist() == [int(x) for x in g["parents"]]
    np.testing.assert_allclose(o["cum_out"][0], np.array(g["scores_ln2"]) * math.log(2), atol=2e-6)
    assert o["slot_out"][0, :, 0].tolist() == [0, 1, 2]


def test_lse_closed_forms():
    V = 151936
    for c in (-3.25, 0.0, 7.5):
        assert abs(osel.lse64(np.full(V, c, F32)) - (c + math.log(V))) < 1e-9
    p = np.random.default_rng(0).dirichlet(np.ones(1000))
    assert abs(osel.lse64(np.log(p))) < 1e-12
    x = np.random.default_rng(1).normal(0, 2, 5000).astype(F32)
    assert abs(osel.lse64(x) - scipy.special.logsumexp(x.astype(np.float64))) < 1e-10


def _round_f32(fr: Fraction) -> F32:
    """Round an exact rational to float32, nearest-even (via an exact fp64 step
    when the rational is a float64, which holds for the cases below)."""
    d = float(fr)
    assert Fraction(d) == fr, "case must be exact in float64"
    return F32(d)


def test_score_is_two_roundings_in_order():
    # cases where fl(cum + fl(x - lse)) differs from one rounding of the exact sum
    rng = np.random.default_rng(3)
    diffs = 0
    for _ in range(2000):
        x = F32(rng.normal(0, 2))
        lse = F32(rng.normal(14, 1))
        cum = F32(-abs(rng.normal(0, 8)))
        lp = _round_f32(Fraction(float(x)) - Fraction(float(lse)))
        want = _round_f32(Fraction(float(cum)) + Fraction(float(lp)))
        got = osel.candidate_scores(np.array([x]), cum, lse)[0]
        assert got == want
        once = _round_f32(Fraction(float(cum)) + Fraction(float(x)) - Fraction(float(lse)))
        diffs += int(once != want)
    assert diffs > 0   # the cases do exercise the double rounding


def _tiny_random_case(seed, levels=True, quantise=False):
    wl = synth.WORKLOADS["tiny"]
    rng = np.random.default_rng(seed)
    items = synth.catalog(wl)
    trie = otrie.build_trie(items, wl.C) if levels else None
    W = 8
    logits = rng.normal(0, 2, size=(1, W, wl.V)).astype(F32)
    if quantise:                       # many exact ties
        logits = np.round(logits).astype(F32)
    cum = np.sort(-np.abs(rng.normal(0, 3, size=(1, W))).astype(F32))[:, ::-1].copy()
    if quantise:
        cum[:] = F32(-1.0)
    level = 1
    pre = items[rng.integers(0, len(items), size=W), :level]
    node = np.array([[trie.node_of_prefix(p) if trie else 0 for p in pre]])
    return wl, trie, logits, cum, node, level


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("use_trie", [True, False])
@pytest.mark.parametrize("quantise", [False, True])
@pytest.mark.parametrize("K", [1, 3, 8, 40])
def test_two_stage_equals_bruteforce(seed, use_trie, quantise, K):
    wl, trie, logits, cum, node, level = _tiny_random_case(seed, use_trie, quantise)
    W = 8
    n_live = np.array([W])
    o = osel.beam_select(logits, cum, node, n_live, np.full((1, W, 3), -1, np.int32),
                         trie, wl.token_base(), level, level, W, K)
    bf = osel.beam_select_bruteforce(logits, cum, node, n_live, trie, wl.token_base(), level, W, K)[0]
    n = o["n_live_out"][0]
    assert n == len(bf)
    assert o["tokens"][0, :n].tolist() == [x[0] for x in bf]
    assert o["parents"][0, :n].tolist() == [x[1] for x in bf]
    assert o["cum_out"][0, :n].tolist() == [float(x[2]) for x in bf]
    assert o["node_out"][0, :n].tolist() == [x[3] for x in bf]


@pytest.mark.parametrize("seed", range(3))
def test_width1_is_greedy_masked_argmax(seed):
    wl, trie, logits, cum, node, level = _tiny_random_case(seed)
    o = osel.beam_select(logits[:, :1], cum[:, :1], node[:, :1], np.array([1]),
                         np.full((1, 1, 3), -1, np.int32), trie, wl.token_base(), level, level, 1, 5)
    codes, _ = trie.children(level, int(node[0, 0]))
    toks = wl.token_base()[level] + codes
    best = toks[np.argmax(logits[0, 0, toks])]       # first max = lowest token on ties
    assert o["tokens"][0, 0] == best and o["parents"][0, 0] == 0


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("use_trie", [True, False])
def test_topk_at_least_width_equals_full_pool(seed, use_trie):
    wl, trie, logits, cum, node, level = _tiny_random_case(seed, use_trie)
    W = 8
    args = (logits, cum, node, np.array([W]), np.full((1, W, 3), -1, np.int32), trie,
            wl.token_base(), level, level, W)
    a = osel.beam_select(*args, W)
    b = osel.beam_select(*args, wl.V)
    for k in ("tokens", "parents", "cum_out", "node_out", "n_live_out"):
        assert np.array_equal(a[k], b[k])


def test_chain_invariants_and_illegal_rate_zero():
    wl = synth.WORKLOADS["tiny"]
    items = synth.catalog(wl)
    outs, hist, trie = _chain(wl, items, lambda t, h, nl: synth.logits(wl, t).numpy())
    catalog = {tuple(x) for x in items.tolist()}
    tb = wl.token_base()
    for t, o in enumerate(outs):
        n = o["n_live_out"][0]
        assert n == min(wl.W, n)
        s = o["cum_out"][0, :n].astype(np.float64)
        key = list(zip(-s, o["parents"][0, :n], o["tokens"][0, :n]))
        assert key == sorted(key)                               # rank order
        prev_live = 1 if t == 0 else outs[t - 1]["n_live_out"][0]
        assert (o["parents"][0, :n] < prev_live).all()
        assert (o["slot_out"][0, :n, t] == t * wl.W + np.arange(n)).all()
        if t > 0:
            prev = outs[t - 1]["slot_out"][0]
            assert (o["slot_out"][0, :n, :t] == prev[o["parents"][0, :n], :t]).all()
    final = outs[-1]
    for j in range(final["n_live_out"][0]):
        codes = tuple(int(tok - tb[lv]) for lv, tok in enumerate(hist[0][j]))
        assert codes in catalog                                 # illegal rate 0
        leaf = sorted(catalog).index(codes)
        assert final["node_out"][0, j] == leaf


def test_exhaustive_catalog_ranking():
    """W >= catalog size and top_k >= codes per level: beam search keeps every
    item, ranked by its float32 cumulative log-probability (logits depend only on
    the prefix, so each item's score is a fixed chain)."""
    wl = synth.WORKLOADS["tiny"]
    items = synth.catalog(wl)
    W = len(items)
    tb = wl.token_base()

    def row_for(prefix_tokens):
        h = hash(tuple(prefix_tokens)) & 0xFFFFFFFF
        return np.random.default_rng(h).normal(0, 2, wl.V).astype(F32)

    def logit_fn(t, hist, n_live):
        lg = np.zeros((1, max(1, int(n_live[0])), wl.V), F32)
        for j in range(int(n_live[0])):
            lg[0, j] = row_for(hist[0][j])
        return lg

    outs, hist, _ = _chain(wl, items, logit_fn, W=W, K=wl.C)
    final = outs[-1]
    assert final["n_live_out"][0] == W
    want = []
    for it in items.tolist():
        cum, prefix = F32(0.0), []
        for lv, c in enumerate(it):
            row = row_for(prefix)
            lse = F32(osel.lse64(row))
            tok = int(tb[lv] + c)
            cum = F32(cum + F32(row[tok] - lse))
            prefix.append(tok)
        want.append((-float(cum), tuple(prefix)))
    want.sort()
    got = [(-float(final["cum_out"][0, j]), tuple(hist[0][j])) for j in range(W)]
    assert [g[1] for g in got] == [w[1] for w in want]
    assert [g[0] for g in got] == [w[0] for w in want]


def test_ties_break_on_beam_then_token():
    V, W = 16, 5
    logits = np.zeros((1, 3, V), F32)      # every score equal
    o = osel.beam_select(logits, np.zeros((1, W), F32), np.zeros((1, W), np.int64),
                         np.array([3]), np.full((1, W, 1), -1, np.int32), None, None, 0, 0, W, 2)
    assert o["parents"][0].tolist() == [0, 0, 1, 1, 2]
    assert o["tokens"][0].tolist() == [0, 1, 0, 1, 0]


def test_fewer_candidates_than_width():
    wl = synth.WORKLOADS["tiny"]
    items = np.array([[1, 2, 3], [1, 2, 4]], np.int32)
    trie = otrie.build_trie(items, wl.C)
    logits = np.random.default_rng(0).normal(0, 2, (1, 8, wl.V)).astype(F32)
    o = osel.beam_select(logits, np.zeros((1, 8), F32), np.zeros((1, 8), np.int64), np.array([1]),
                         np.full((1, 8, 3), -1, np.int32), trie, wl.token_base(), 0, 0, 8, 8)
    assert o["n_live_out"][0] == 1
    assert o["tokens"][0, 1:].tolist() == [-1] * 7
    assert np.isneginf(o["cum_out"][0, 1:]).all()
