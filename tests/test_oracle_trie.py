"""Pins for the oracle's catalog trie (CPU only)."""
import numpy as np
import pytest

import synth
from oracle import trie as otrie
from tests.golden import read_kv


def test_golden_small_trie():
    g = read_kv("trie_small.txt")
    items = np.array(g["items"], dtype=np.int32)
    t = otrie.build_trie(items, 4)
    for lv in range(3):
        assert t.off[lv].tolist() == [int(x) for x in g[f"off{lv}"]]
        assert t.code[lv].tolist() == [int(x) for x in g[f"code{lv}"]]
        assert t.child_node[lv].tolist() == [int(x) for x in g[f"child{lv}"]]
    assert t.items.tolist() == g["leaves"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_dict_builder(seed):
    rng = np.random.default_rng(seed)
    items = rng.integers(0, 5, size=(60, 3)).astype(np.int32)   # many duplicates
    t = otrie.build_trie(items, 5)
    off, code, child = otrie.build_trie_dict(items.tolist(), 5)
    for lv in range(3):
        assert np.array_equal(t.off[lv], off[lv])
        assert np.array_equal(t.code[lv], code[lv])
        assert np.array_equal(t.child_node[lv], child[lv])


def test_tiny_catalog_round_trip():
    wl = synth.WORKLOADS["tiny"]
    items = synth.catalog(wl)
    assert len({tuple(x) for x in items.tolist()}) == wl.n_items   # distinct by construction
    t = otrie.build_trie(items, wl.C)
    off, code, child = otrie.build_trie_dict(items.tolist(), wl.C)
    for lv in range(wl.levels):
        assert np.array_equal(t.off[lv], off[lv])
        assert np.array_equal(t.code[lv], code[lv])
    # every item reaches a leaf; the leaf number is its rank among sorted items
    srt = sorted(map(tuple, items.tolist()))
    rank = {it: i for i, it in enumerate(srt)}
    for it in items.tolist():
        assert t.node_of_prefix(it) == rank[tuple(it)]
    assert t.n_nodes(wl.levels - 1) <= len(srt)
    assert len(t.code[wl.levels - 1]) == len(srt)          # leaf count = distinct items
    # absent prefixes are rejected
    absent = next(p for p in ((a, b, c) for a in range(16) for b in range(16) for c in range(16))
                  if p not in rank)
    assert t.node_of_prefix(absent) == -1


def test_zipf_catalog_shape():
    wl = synth.WORKLOADS["qwen06b"].scaled(n_items=20000)
    items = synth.catalog(wl)
    assert items.shape == (20000, 3)
    assert len(np.unique(items, axis=0)) == 20000
    assert items.min() >= 0 and items.max() < wl.C
    # Zipf(1.1): code 0 is the most frequent at every level
    for lv in range(3):
        cnt = np.bincount(items[:, lv], minlength=wl.C)
        assert cnt.argmax() == 0
