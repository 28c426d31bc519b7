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


def test_static_scratch_matches_the_oracle(gpu_lib):
    """Two calls in a row given the oracle's float32 normalisers (lse_in): the
    selections equal the oracle's bit for bit."""
    from oracle import select as osel
    from tests._helpers import build_tries, compare_select, oracle_lse32
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"].scaled(n_items=200_000)
    gtrie, otr = build_tries(wl, synth.catalog(wl))
    st = _state(wl.R, wl.W, wl.T)
    o_cum, o_node = np.zeros((wl.R, wl.W), np.float32), np.zeros((wl.R, wl.W), np.int64)
    o_nl, o_slot = np.ones(wl.R, np.int32), np.full((wl.R, wl.W, wl.T), -1, np.int32)
    for t in range(2):
        lg = synth.logits(wl, t, device=DEV)
        lg_np = lg.cpu().numpy()
        lse32 = oracle_lse32(lg_np, o_nl)
        got = bd.beam_select_static(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, t, t, wl.K,
                                    lse_in=torch.from_numpy(np.nan_to_num(lse32)).to(DEV))
        ref = osel.beam_select(lg_np, o_cum, o_node, o_nl, o_slot, otr, wl.token_base(), t, t, wl.W, wl.K,
                               lse32=lse32)
        compare_select(got, ref, t, f"static step {t}")
        st = dict(cum=got["cum_out"], node=got["node_out"], n_live=got["n_live_out"], slot=got["slot_out"])
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]


def test_static_scratch_allocates_nothing(gpu_lib):
    """After a first call (which resolves the array's address), further calls
    with preallocated outputs leave the device's free memory unchanged."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["openvocab"].scaled(W=64, K=64, T=2)
    st = _state(wl.R, wl.W, wl.T)
    st["n_live"].fill_(wl.W)
    lg = synth.logits(wl, 0, device=DEV)
    out = dict(tokens=torch.empty((wl.R, wl.W), dtype=torch.int32, device=DEV),
               parents=torch.empty((wl.R, wl.W), dtype=torch.int32, device=DEV),
               cum_out=torch.empty((wl.R, wl.W), dtype=torch.float32, device=DEV),
               lse_out=torch.empty((wl.R, wl.W), dtype=torch.float32, device=DEV),
               node_out=torch.empty((wl.R, wl.W), dtype=torch.int32, device=DEV),
               n_live_out=torch.empty((wl.R,), dtype=torch.int32, device=DEV),
               slot_out=torch.empty((wl.R, wl.W, wl.T), dtype=torch.int32, device=DEV))
    bd.beam_select_static(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, 1, wl.K, out=out)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        bd.beam_select_static(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, 1, wl.K, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(out["n_live_out"].min()) == wl.W
