"""The whole T-step decode chain replayed as one CUDA graph (DecodeChain).

The graph holds the same launches as the eager calls, so every output of
every step must equal the eager chain's bit for bit, on the first replay
and on later ones (each replay restarts from one live beam per request).
"""
import pytest
import torch

import synth

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
