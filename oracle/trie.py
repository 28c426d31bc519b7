"""Catalog trie in canonical CSR form (oracle side).

Items are semantic ids: fixed-length tuples of codes, one code per level, each
level a contiguous range of the vocabulary ("Deploying FlashRec": SID layout;
"Generative recommendation design" §4.1.1: each decode step emits one token and
the tokens together form the item id).  Early filtering of invalid items
("Generative recommendation design" §4.3; FlashRec's fused SID trie, dense or
CSR) needs, for every beam, the set of codes that extend its prefix to some
catalog item.

Canonical form (the reading of the pages used throughout):

* items are de-duplicated;
* the nodes of level t are the distinct length-t prefixes, numbered in
  lexicographic order (level 0 holds only the empty prefix, node 0);
* the children of a node are its distinct next codes in ascending order;
* ``child_node[e]`` is the number of the extended prefix among level t+1 nodes;
  for the last level that is the item's index among the distinct sorted items.

Per level t the CSR arrays are ``off`` (n_nodes_t + 1, int64 here) and
``code`` / ``child_node`` (n_edges_t).
"""
from dataclasses import dataclass

import numpy as np


@dataclass
class Trie:
    levels: int
    C: int
    off: list         # per level: int64 [n_nodes_t + 1]
    code: list        # per level: int32 [n_edges_t]
    child_node: list  # per level: int64 [n_edges_t]
    items: np.ndarray  # distinct items, lexicographic order [n_distinct, levels]

    def n_nodes(self, t):
        return len(self.off[t]) - 1

    def children(self, t, node):
        """(codes, child nodes) of ``node`` at level t."""
        a, b = int(self.off[t][node]), int(self.off[t][node + 1])
        return self.code[t][a:b], self.child_node[t][a:b]

    def node_of_prefix(self, prefix):
        """Walk codes from the root; returns the node id or -1 if absent."""
        node = 0
        for t, c in enumerate(prefix):
            codes, kids = self.children(t, node)
            pos = np.searchsorted(codes, c)
            if pos >= len(codes) or codes[pos] != c:
                return -1
            node = int(kids[pos])
        return node


def _prefix_keys(items: np.ndarray, t: int, C: int) -> np.ndarray:
    """Integer key of each item's length-t prefix; integer order = lexicographic."""
    k = np.zeros(items.shape[0], dtype=np.int64)
    for lv in range(t):
        k = k * C + items[:, lv].astype(np.int64)
    return k


def build_trie(items: np.ndarray, C: int) -> Trie:
    """Canonical CSR trie of a catalog ``items`` [n, levels] (codes in [0, C)).

    Pinned by a dictionary-of-sets builder and a leaf round trip in the tests.
    """
    items = np.asarray(items, dtype=np.int64)
    levels = items.shape[1]
    nodes = [np.unique(_prefix_keys(items, t, C)) for t in range(levels + 1)]
    off, code, child = [], [], []
    for t in range(levels):
        ext = nodes[t + 1]                      # every edge is a distinct (t+1)-prefix
        parent = np.searchsorted(nodes[t], ext // C)
        counts = np.bincount(parent, minlength=len(nodes[t]))
        off.append(np.concatenate([[0], np.cumsum(counts)]).astype(np.int64))
        code.append((ext % C).astype(np.int32))
        child.append(np.searchsorted(nodes[t + 1], ext).astype(np.int64))
    distinct = np.zeros((len(nodes[levels]), levels), dtype=np.int32)
    k = nodes[levels].copy()
    for lv in reversed(range(levels)):
        distinct[:, lv] = k % C
        k //= C
    return Trie(levels, C, off, code, child, distinct)


def build_trie_dict(items, C):
    """Second, independent builder (nested dicts of sets), used only to pin
    ``build_trie`` on small catalogs."""
    levels = len(items[0]) if len(items) else 0
    prefixes = [sorted({tuple(int(c) for c in it[:t]) for it in items}) for t in range(levels + 1)]
    index = [{p: i for i, p in enumerate(ps)} for ps in prefixes]
    off, code, child = [], [], []
    for t in range(levels):
        kids = {p: set() for p in prefixes[t]}
        for p in prefixes[t + 1]:
            kids[p[:-1]].add(p[-1])
        o, cs, ch = [0], [], []
        for p in prefixes[t]:
            for c in sorted(kids[p]):
                cs.append(c)
                ch.append(index[t + 1][p + (c,)])
            o.append(len(cs))
        off.append(np.array(o, dtype=np.int64))
        code.append(np.array(cs, dtype=np.int32))
        child.append(np.array(ch, dtype=np.int64))
    return off, code, child
