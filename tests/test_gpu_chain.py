"""The whole T-step decode chain replayed as one CUDA graph (DecodeChain).

The graph holds the same launches as the eager calls, so every output of
every step must equal the eager chain's bit for bit, on the first replay
and on later ones (each replay restarts from one live beam per request).
The graph is also tied to the oracle: replayed with every step's candidates
scored against the oracle's float32 normalisers, each step's selection equals
the oracle's chain bit for bit, and each step's attention output, computed
over the slot rows the chain's own selection produced, matches the float64
oracle within the bf16 tolerance on beams from every 256-row tile of the
tensor-core shared stage.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import select as osel
from tests._helpers import ATOL_ATTN, build_tries, compare_select, oracle_attn_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(wl):
    from wide_beam_generative_gb300 import beamdec as bd
    items = synth.catalog(wl)
    trie = bd.beam_trie_build(items, [wl.C] * wl.levels, wl.token_base(), wl.V) if wl.levels else None
    att = [synth.attention_inputs(wl, t, device=DEV) for t in range(wl.T)]
    logits = [synth.logits(wl, t, device=DEV) for t in range(wl.T)]
    return trie, att, logits


def _eager(wl, trie, att, logits):
    from wide_beam_generative_gb300 import beamdec as bd
    R, W, T = wl.R, wl.W, wl.T
    a0 = att[0]
    maxp = int(synth.prompt_lens(wl).max())
    st = dict(cum=torch.zeros((R, W), dtype=torch.float32, device=DEV),
              node=torch.zeros((R, W), dtype=torch.int32, device=DEV),
              n_live=torch.ones((R,), dtype=torch.int32, device=DEV),
              slot=torch.full((R, W, T), -1, dtype=torch.int32, device=DEV))
    outs = []
    for t in range(T):
        o = bd.beam_select(logits[t], st["cum"], st["node"], st["n_live"], st["slot"], trie, t, t, wl.K)
        y = bd.beam_attn_decode(att[t]["q"], a0["shared_k"], a0["shared_v"], a0["prompt_offsets"], maxp,
                                a0["unshared_k"], a0["unshared_v"], o["slot_out"], o["n_live_out"], t,
                                k_scale=a0["k_scale"], v_scale=a0["v_scale"])
        outs.append((o, y))
        st = dict(cum=o["cum_out"], node=o["node_out"], n_live=o["n_live_out"], slot=o["slot_out"])
    return outs


@pytest.mark.parametrize("name", ["qwen06b", "onerec17b"])
def test_graph_chain_equals_eager(gpu_lib, name):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS[name]
    trie, att, logits = _inputs(wl)
    ref = _eager(wl, trie, att, logits)
    a0 = att[0]
    chain = bd.DecodeChain(logits, [a["q"] for a in att], a0["shared_k"], a0["shared_v"],
                           a0["prompt_offsets"], int(synth.prompt_lens(wl).max()), a0["unshared_k"],
                           a0["unshared_v"], trie, wl.K, k_scale=a0["k_scale"], v_scale=a0["v_scale"])
    for rep in range(2):
        for t in range(wl.T):   # scribble over the outputs so a replay that skipped a step would show
            chain.out[t].fill_(7)
            chain.sel[t]["tokens"].fill_(-7)
        chain.replay()
        torch.cuda.synchronize()
        assert chain.status() == (0, 0)
        for t in range(wl.T):
            o, y = ref[t]
            for k in ("tokens", "parents", "cum_out", "node_out", "n_live_out", "slot_out"):
                assert torch.equal(chain.sel[t][k], o[k]), (rep, t, k)
            assert torch.equal(chain.out[t], y), (rep, t)


def _tile_beams(wl):
    """Beams whose query rows fall in every 256-row tile of the shared stage
    (rows j*G .. j*G + G-1 of beam j): the first and last beam of each tile."""
    per = max(1, 256 // wl.G)
    beams = set()
    for j0 in range(0, wl.W, per):
        beams.update({j0, min(wl.W, j0 + per) - 1})
    return sorted(beams)


@pytest.mark.parametrize("name", ["qwen06b", "onerec17b"])
def test_graph_chain_matches_oracle(gpu_lib, name):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS[name]
    items = synth.catalog(wl)
    trie, otr = build_tries(wl, items)
    att = [synth.attention_inputs(wl, t, device=DEV) for t in range(wl.T)]
    logits = [synth.logits(wl, t, device=DEV) for t in range(wl.T)]
    lg_np = [lg.cpu().numpy() for lg in logits]
    # the oracle's float64 normaliser of every row, rounded to float32
    lse32 = [np.array([[osel.lse64(x[r, b]) for b in range(wl.W)] for r in range(wl.R)], np.float32)
             for x in lg_np]
    a0 = att[0]
    chain = bd.DecodeChain(logits, [a["q"] for a in att], a0["shared_k"], a0["shared_v"],
                           a0["prompt_offsets"], int(synth.prompt_lens(wl).max()), a0["unshared_k"],
                           a0["unshared_v"], trie, wl.K, k_scale=a0["k_scale"], v_scale=a0["v_scale"],
                           score_lse=[torch.from_numpy(x).to(DEV) for x in lse32])
    chain.replay()
    torch.cuda.synchronize()
    assert chain.status() == (0, 0)
    R, W, T = wl.R, wl.W, wl.T
    o_cum, o_node = np.zeros((R, W), np.float32), np.zeros((R, W), np.int64)
    o_nl, o_slot = np.ones(R, np.int32), np.full((R, W, T), -1, np.int32)
    beams = _tile_beams(wl)
    for t in range(T):
        ref = osel.beam_select(lg_np[t], o_cum, o_node, o_nl, o_slot, otr, wl.token_base(), t, t, W, wl.K,
                               lse32=lse32[t])
        compare_select(chain.sel[t], ref, t, f"graph {name} step {t}")
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]
        # attention over the chain's slot rows (equal to the oracle's, checked above)
        inp = oracle_attn_inputs(a0, att[t]["q"], wl)
        todo = [(r, j) for r in range(R) for j in beams if j < int(o_nl[r])]
        want = oatt.attention_decode(inp, o_slot, o_nl, t, beams=todo)
        got = chain.out[t].double().cpu().numpy()
        err = max(float(np.abs(got[r, j] - want[r, j]).max()) for r, j in todo)
        assert err < ATOL_ATTN[wl.kv_dtype], (t, err)
        dead = [(r, j) for r in range(R) for j in range(int(o_nl[r]), W)]
        for r, j in dead[:8]:
            assert not np.any(got[r, j]), (t, r, j)


@pytest.mark.parametrize("prompt", [128, 1024])   # one prompt split (fused merge) / several (merge kernel)
def test_eager_chain_with_dead_tiles_matches_oracle(gpu_lib, prompt):
    """A catalog of 40 items leaves at most 40 of 300 beams alive after the
    first steps, so whole 256-row tiles of the shared stage are dead while
    the attention, launched right behind the selection that produced its
    slot rows and live counts, reads them only after that selection has
    completed.  Every step's attention, over the selection's own outputs,
    matches the float64 oracle on live beams and is zero on dead ones."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"].scaled(name="deadtiles", W=300, K=300, n_items=40,
                                           prompt_lens=[prompt], T=3)
    trie, att, logits = _inputs(wl)
    outs = _eager(wl, trie, att, logits)
    torch.cuda.synchronize()
    a0 = att[0]
    R, W, T = wl.R, wl.W, wl.T
    beams = _tile_beams(wl)
    saw_dead_tile = False
    for t in range(T):
        o, y = outs[t]
        nl = o["n_live_out"].cpu().numpy()
        slot = o["slot_out"].cpu().numpy()
        saw_dead_tile |= t > 0 and int(nl.min()) * wl.G <= 256 and W * wl.G > 512
        inp = oracle_attn_inputs(a0, att[t]["q"], wl)
        todo = [(r, j) for r in range(R) for j in beams + list(range(min(W, 4))) if j < int(nl[r])]
        want = oatt.attention_decode(inp, slot, nl, t, beams=todo)
        got = y.double().cpu().numpy()
        err = max(float(np.abs(got[r, j] - want[r, j]).max()) for r, j in todo)
        assert err < ATOL_ATTN[wl.kv_dtype], (t, err)
        for r in range(R):
            assert not np.any(got[r, int(nl[r]):]), (t, r)
    assert saw_dead_tile
