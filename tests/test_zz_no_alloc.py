"""beam_select_static (no workspace, no allocation) against beam_select.

The static variant is for callers that cannot allocate device memory, such as
a plugin interface that only hands the library its inputs and outputs.  Its
results must equal those of beam_select with a caller-owned workspace, bit for
bit (the tolerance of every selection test), on two calls in a row that share
the static scratch array.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _state(R, W, T):
    return dict(cum=torch.zeros((R, W), dtype=torch.float32, device=DEV),
                node=torch.zeros((R, W), dtype=torch.int32, device=DEV),
                n_live=torch.ones((R,), dtype=torch.int32, device=DEV),
                slot=torch.full((R, W, T), -1, dtype=torch.int32, device=DEV))


def _same(a, b, live_rows):
    for k in ("tokens", "parents", "cum_out", "node_out", "n_live_out", "slot_out"):
        assert torch.equal(a[k], b[k]), k
    for r, n in enumerate(live_rows):
        assert torch.equal(a["lse_out"][r, :n], b["lse_out"][r, :n])


def test_static_scratch_matches_workspace_path(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"].scaled(R=2, n_items=200_000)
    items = synth.catalog(wl)
    trie = bd.beam_trie_build(items, [wl.C] * wl.levels, wl.token_base(), wl.V)
    st = _state(wl.R, wl.W, wl.T)
    for t in range(2):                       # two calls in a row on the shared array
        lg = synth.logits(wl, t, device=DEV)
        live = st["n_live"].cpu().tolist()
        ref = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], trie, t, t, wl.K)
        got = bd.beam_select_static(lg, st["cum"], st["node"], st["n_live"], st["slot"], trie, t, t, wl.K)
        torch.cuda.synchronize()
        _same(ref, got, live)
        st = dict(cum=got["cum_out"], node=got["node_out"], n_live=got["n_live_out"], slot=got["slot_out"])
    assert int(st["n_live"].min()) == wl.W


def test_static_scratch_open_vocab_and_size_limit(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["openvocab"].scaled(W=40, K=40, T=2)
    st = _state(wl.R, wl.W, wl.T)
    for t in range(2):
        lg = synth.logits(wl, t, device=DEV)
        live = st["n_live"].cpu().tolist()
        ref = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, t, wl.K)
        got = bd.beam_select_static(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, t, wl.K)
        torch.cuda.synchronize()
        _same(ref, got, live)
        st = dict(cum=got["cum_out"], node=got["node_out"], n_live=got["n_live_out"], slot=got["slot_out"])
    # a shape whose scratch exceeds the static array is refused before any launch
    import ctypes
    fake = ctypes.c_void_p(0x1000)
    rc = bd.lib().beam_select_static(fake, 151936, None, fake, fake, fake, fake, None, 0, 0,
                                     2, 5000, 5000, 151936, 2, fake, fake, fake, None, fake, fake,
                                     ctypes.c_void_p(0x2000), None)
    assert rc == bd.ERR_UNSUPPORTED
