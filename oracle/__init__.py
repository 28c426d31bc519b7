"""CPU oracle for the wide-beam decode step (TEST INFRASTRUCTURE ONLY).

A plain, slow, float64 restatement of what the decode step computes, written
from the pages that describe the method:

* "Generative recommendation design" (xLLM documentation), §4.1.1 (beam
  expansion over a beam_width x top_k pool), §4.2.1 (shared prompt KV stored
  once, unshared decode-token KV per beam), §4.2.2 (shared stage, unshared
  stage, online-softmax merge), §4.3 (filter invalid items early), §6 (beam
  search followed by cache selection after the reorder).
* SGLang pull request 31626 (per-request beam search) and the FlashRec
  announcement in the same thread: beam rows alias the leader's prompt KV; a
  catalog trie keeps every continuation a valid semantic id.
* "Deploying FlashRec": temperature 0 is deterministic top-k; the returned
  sequence score is the cumulative log-probability.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
library and its Python binding never call it; the oracle shares no code,
header, table or helper with the CUDA path.

Modules
-------
``trie``       canonical CSR catalog trie (``build_trie``)
``select``     log-softmax + trie mask + per-beam top_k + global top-W
``attention``  attention over the explicitly concatenated prompt + ancestor KV
``dequant``    exact decoding of bf16 / e4m3 bytes to float64

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
brute force and invariants; see the docstring of each function for its pin.
"""
from . import attention, dequant, select, trie  # noqa: F401
