"""GPU parity of beam_trie_build and beam_select against the CPU oracle.

Selection is compared bit for bit (tokens, parents, scores, child nodes, slot
rows, live counts) when both sides use the same float32 log-sum-exp (the
oracle's float64 value rounded to float32, passed to the kernel through
``lse_in``).  The kernel's own log-sum-exp is compared with the oracle's
float64 value within 1e-5, and the full path (kernel computes its own
normaliser) is compared with a tolerance only at exact near-ties.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import select as osel
from tests._helpers import ATOL_LSE, build_tries, compare_select, oracle_lse32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _catalog(wl):
    return synth.catalog(wl)


def _init_state(R, W, T):
    return dict(cum=torch.zeros((R, W), dtype=torch.float32, device=DEV),
                node=torch.zeros((R, W), dtype=torch.int32, device=DEV),
                n_live=torch.ones((R,), dtype=torch.int32, device=DEV),
                slot=torch.full((R, W, T), -1, dtype=torch.int32, device=DEV))


def run_chain(wl, items=None, steps=None, K=None, W=None, logit_fn=None, check=True, temperature=0.0,
              seed=0, dense_levels=()):
    """Decode `steps` steps on the GPU and in the oracle in lockstep
    (temperature > 0: Gumbel top-k under `seed` on both sides)."""
    from wide_beam_generative_gb300 import beamdec as bd
    W = W or wl.W
    K = K or wl.K
    T = wl.T
    steps = T if steps is None else steps
    if wl.levels:
        gtrie, otr = build_tries(wl, items)
        for lv in dense_levels:
            gtrie.make_dense(lv)
    else:
        gtrie, otr = None, None
    st = _init_state(wl.R, W, T)
    o_cum = np.zeros((wl.R, W), np.float32)
    o_node = np.zeros((wl.R, W), np.int64)
    o_nl = np.ones(wl.R, np.int32)
    o_slot = np.full((wl.R, W, T), -1, np.int32)
    ws = bd.workspace(bd.beam_select_workspace_size(wl.R, W, K, wl.V))
    outs = []
    for t in range(steps):
        lg = logit_fn(t) if logit_fn else synth.logits(wl.scaled(W=W), t, device=DEV)
        lg_np = lg.cpu().numpy()
        lse32 = oracle_lse32(lg_np, o_nl)
        res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, t, t, K,
                             lse_in=torch.from_numpy(np.nan_to_num(lse32)).to(DEV), ws=ws,
                             temperature=temperature, seed=seed)
        ref = osel.beam_select(lg_np, o_cum, o_node, o_nl, o_slot, otr, wl.token_base(), t, t, W, K,
                               lse32=lse32, temperature=temperature, seed=seed)
        if check:
            compare_select(res, ref, t, f"{wl.name} step {t}")
        assert bd.read_status(ws) == 0
        outs.append((res, ref))
        st = dict(cum=res["cum_out"], node=res["node_out"], n_live=res["n_live_out"], slot=res["slot_out"])
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]
    return outs


# ---------------------------------------------------------------------------- trie

@pytest.mark.parametrize("name,n_items", [("tiny", None), ("qwen06b", None), ("fp8kv", 200_000)])
def test_trie_matches_oracle(gpu_lib, name, n_items):
    wl = synth.WORKLOADS[name]
    if n_items:
        wl = wl.scaled(n_items=n_items)
    items = _catalog(wl)
    gtrie, otr = build_tries(wl, items)
    info = gtrie.info()
    assert info["n_items"] == len(otr.items)
    for lv in range(wl.levels):
        off, code = gtrie.export(lv)
        assert np.array_equal(off.cpu().numpy(), otr.off[lv])
        assert np.array_equal(code.cpu().numpy(), otr.code[lv])
        # canonical numbering: the child reached by edge e is node e of the next level
        assert np.array_equal(otr.child_node[lv], np.arange(len(otr.code[lv])))
        assert info["max_children"][lv] == int(np.diff(otr.off[lv]).max())


def test_trie_with_duplicates_and_unsorted_input(gpu_lib):
    from tests.golden import read_kv
    from oracle import trie as otrie
    from wide_beam_generative_gb300 import beamdec as bd
    g = read_kv("trie_small.txt")
    items = np.array(g["items"], np.int32)
    t = bd.beam_trie_build(items, [4, 4, 4], [0, 4, 8], 12)
    for lv in range(3):
        off, code = t.export(lv)
        assert off.cpu().tolist() == [int(x) for x in g[f"off{lv}"]]
        assert code.cpu().tolist() == [int(x) for x in g[f"code{lv}"]]
    assert t.info()["n_items"] == 6


# ---------------------------------------------------------------------------- lse

def test_lse_matches_float64(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"].scaled(W=64, K=4, levels=0, n_items=0)
    lg = synth.logits(wl, 0, device=DEV)                       # N(0, 2)
    lg[0, 1] = 3.25                                            # constant row: lse = c + ln V
    lg[0, 2] = synth.logits(synth.WORKLOADS["fp8kv"].scaled(W=64), 1, device=DEV)[0, 2]  # spikes
    lg[0, 3, 5] = 60.0                                         # one dominant logit
    R, W, V = 1, 64, wl.V
    st = _init_state(R, W, 1)
    st["n_live"][:] = W
    res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, 0, 4)
    got = res["lse_out"].cpu().numpy()[0].astype(np.float64)
    lg_np = lg.cpu().numpy()
    want = np.array([osel.lse64(lg_np[0, b]) for b in range(W)])
    assert np.abs(got - want).max() < ATOL_LSE
    assert abs(got[1] - (3.25 + np.log(V))) < ATOL_LSE


# ---------------------------------------------------------------------------- selection, bit-exact

def test_tiny_chain_bitexact(gpu_lib):
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl, _catalog(wl))


@pytest.mark.parametrize("K", [1, 3, 8, 20])
@pytest.mark.parametrize("W", [1, 8, 37])
def test_tiny_chain_widths(gpu_lib, K, W):
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl.scaled(W=W), _catalog(wl), K=K, W=W)


def test_tiny_open_vocab_with_ties(gpu_lib):
    wl = synth.WORKLOADS["tiny"].scaled(name="tiny-open", levels=0, n_items=0, W=16)

    def quantised(t):   # integer logits: many exact ties in score
        return torch.round(synth.logits(wl, t, device=DEV))
    run_chain(wl, None, K=5, W=16, logit_fn=quantised)


def test_constant_logits_all_ties(gpu_lib):
    wl = synth.WORKLOADS["tiny"].scaled(name="tiny-const", levels=0, n_items=0, W=12)
    run_chain(wl, None, K=7, W=12, logit_fn=lambda t: torch.zeros((1, 12, wl.V), device=DEV))


def test_qwen06b_chain_bitexact(gpu_lib):
    wl = synth.WORKLOADS["qwen06b"]
    run_chain(wl, _catalog(wl))


def test_open_vocab_large_vocab(gpu_lib):
    wl = synth.WORKLOADS["openvocab"].scaled(W=48, K=48, T=4)
    run_chain(wl, None, steps=3)
    run_chain(wl, None, steps=2, K=5)          # top_k < beam_width: per-beam cap binds


def test_onerec17b_full_size_bitexact(gpu_lib):
    """The benchmarked workload at full size: 4 requests x 512 beams, top_k 512,
    4M-item Zipf catalog, vocab 151936, all three steps."""
    wl = synth.WORKLOADS["onerec17b"]
    outs = run_chain(wl, _catalog(wl))
    assert int(outs[-1][0]["n_live_out"].min()) == wl.W


def test_fp8kv_full_size_bitexact(gpu_lib):
    """4 requests x 1000 beams, top_k 128 < W, 4 SID levels of 4096, 2M items,
    logits N(0,3) with 1% spikes of +8."""
    wl = synth.WORKLOADS["fp8kv"]
    run_chain(wl, _catalog(wl))


def test_openvocab_full_size_properties(gpu_lib):
    """2 requests x 5000 beams, top_k 5000, open vocabulary 151936: 25M-candidate
    pools.  Step 0 is compared bit for bit; step 1 is checked exactly without a
    full sort: with top_k >= W the selection is the top-W of the whole pool, so
    the count of candidates whose key is at or below the W-th selected key must
    be exactly W, and every selected score must equal its recomputed value."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["openvocab"]
    outs = run_chain(wl, None, steps=1)
    res0 = outs[0][0]
    R, W, V = wl.R, wl.W, wl.V
    lg = synth.logits(wl, 1, device=DEV)
    lse64 = torch.logsumexp(lg.double(), dim=-1)                      # float64 on device
    lse32 = lse64.float()
    res = bd.beam_select(lg, res0["cum_out"], res0["node_out"], res0["n_live_out"], res0["slot_out"],
                         None, 1, 1, wl.K, lse_in=lse32)
    assert int(res["n_live_out"].min()) == W
    cum_in = res0["cum_out"]
    for r in range(R):
        par = res["parents"][r].long()
        tok = res["tokens"][r].long()
        s_sel = (cum_in[r, par] + (lg[r, par, tok] - lse32[r, par]))
        assert torch.equal(s_sel, res["cum_out"][r])                  # fp32 round-to-nearest steps
        # exact top-W check by counting (score desc, beam asc, token asc) <= W-th key
        sW, bW, tW = res["cum_out"][r, W - 1], int(par[W - 1]), int(tok[W - 1])
        count = 0
        for b0 in range(0, W, 500):
            s = cum_in[r, b0:b0 + 500, None] + (lg[r, b0:b0 + 500] - lse32[r, b0:b0 + 500, None])
            bidx = torch.arange(b0, b0 + s.shape[0], device=DEV)[:, None]
            tidx = torch.arange(V, device=DEV)[None, :]
            better = (s > sW) | ((s == sW) & ((bidx < bW) | ((bidx == bW) & (tidx <= tW))))
            count += int(better.sum())
        assert count == W


# ---------------------------------------------------------------------------- full path

def run_chain_own_lse(wl, steps=None, items=None, temperature=0.0, seed=0, dense_levels=()):
    """The production path (the kernel computes each row's normaliser, so the
    selection runs in the one-launch stream kernel) against the oracle's own
    float64 chain.  Each side carries its own state.  Per step: log-sum-exp
    within 1e-5 of float64; the selected (parent, token, score) rows equal the
    oracle's, except where the two sides' independently rounded normalisers
    reorder near-ties: candidates whose scores lie within 4e-5 of the cut may
    trade places with ones outside, and two selected candidates whose scores
    differ by less than 4e-5 may swap ranks.  After such a difference the
    states differ, so later steps are not compared.  Returns the number of
    steps compared exactly."""
    from wide_beam_generative_gb300 import beamdec as bd
    W, K, R, T = wl.W, wl.K, wl.R, wl.T
    steps = T if steps is None else steps
    gtrie, otr = build_tries(wl, items) if wl.levels else (None, None)
    for lv in dense_levels:
        gtrie.make_dense(lv)
    st = _init_state(R, W, T)
    o_cum = np.zeros((R, W), np.float32)
    o_node = np.zeros((R, W), np.int64)
    o_nl = np.ones(R, np.int32)
    o_slot = np.full((R, W, T), -1, np.int32)
    ws = bd.workspace(bd.beam_select_workspace_size(R, W, K, wl.V))
    exact = 0
    for t in range(steps):
        lg = synth.logits(wl, t, device=DEV)
        res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, t, t, K, ws=ws,
                             temperature=temperature, seed=seed)
        assert bd.read_status(ws) == 0
        ref = osel.beam_select(lg.cpu().numpy(), o_cum, o_node, o_nl, o_slot, otr, wl.token_base(), t, t,
                               W, K, temperature=temperature, seed=seed)
        got_lse = res["lse_out"].cpu().numpy()
        g = {k: res[k].cpu().numpy() for k in ("parents", "tokens", "cum_out", "node_out", "n_live_out",
                                               "slot_out")}
        traded = False
        for r in range(R):
            nl_in = int(o_nl[r])
            assert np.abs(got_lse[r, :nl_in].astype(np.float64) - ref["lse64"][r, :nl_in]).max() < ATOL_LSE
            n = int(ref["n_live_out"][r])
            assert int(g["n_live_out"][r]) == n
            g_s = g["cum_out"][r, :n].astype(np.float64)
            o_s = ref["cum_out"][r, :n].astype(np.float64)
            assert np.abs(g_s - o_s).max() < 2e-5
            same = (np.array_equal(g["parents"][r, :n], ref["parents"][r, :n]) and
                    np.array_equal(g["tokens"][r, :n], ref["tokens"][r, :n]))
            if same:
                assert np.array_equal(g["node_out"][r, :n], ref["node_out"][r, :n])
                assert np.array_equal(g["slot_out"][r, :n], ref["slot_out"][r, :n])
                continue
            traded = True
            cut = o_s[-1]
            g_set = set(zip(g["parents"][r, :n], g["tokens"][r, :n]))
            o_set = set(zip(ref["parents"][r, :n], ref["tokens"][r, :n]))
            lookup = {(p, tk): sc for p, tk, sc in zip(ref["parents"][r, :n], ref["tokens"][r, :n], o_s)}
            for key in g_set ^ o_set:
                if key in lookup:
                    assert abs(lookup[key] - cut) < 4e-5
            # the GPU's order of the selected candidates inverts no pair
            # whose oracle scores differ by 4e-5 or more
            # (a candidate only the GPU selected stands in with its own
            # score, which must lie near the cut as well)
            g_lookup = {(p, tk): sc for p, tk, sc in zip(g["parents"][r, :n], g["tokens"][r, :n], g_s)}
            for key in g_set - o_set:
                assert abs(g_lookup[key] - cut) < 6e-5
            o_score = np.array([lookup.get(key, g_lookup[key])
                                for key in zip(g["parents"][r, :n], g["tokens"][r, :n])])
            assert np.all(np.minimum.accumulate(o_score)[:-1] >= o_score[1:] - 4e-5)
        if traded:
            break
        exact += 1
        st = dict(cum=res["cum_out"], node=res["node_out"], n_live=res["n_live_out"], slot=res["slot_out"])
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]
    return exact


def test_full_path_own_lse(gpu_lib):
    """qwen06b, 3 steps, the one-launch selection against the oracle's chain."""
    wl = synth.WORKLOADS["qwen06b"]
    assert run_chain_own_lse(wl, items=_catalog(wl)) >= 1


def test_onerec17b_full_size_own_lse(gpu_lib):
    """The benchmarked shape (4 x 512 beams, top_k 512) on the production path:
    row expansion in each row's last stream block and the request tail in the
    request's last row, against the oracle's chain."""
    wl = synth.WORKLOADS["onerec17b"]
    assert run_chain_own_lse(wl, items=_catalog(wl)) >= 1


def test_fp8kv_full_size_own_lse(gpu_lib):
    """4 x 1000 beams, top_k 128, four SID levels: more than 1024 candidates at
    or above the cut's bin, so the tail takes the radix-narrowing path."""
    wl = synth.WORKLOADS["fp8kv"]
    assert run_chain_own_lse(wl, items=_catalog(wl)) >= 1


def test_deterministic_repeat(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"]
    items = _catalog(wl)
    gtrie, _ = build_tries(wl, items)
    st = _init_state(wl.R, wl.W, wl.T)
    lg = synth.logits(wl, 0, device=DEV)
    a = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K)
    b = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K)
    for k in a:
        if k == "lse_out":        # written for the live input rows only
            assert torch.equal(a[k][:, :1], b[k][:, :1])
        elif a[k] is not None:
            assert torch.equal(a[k], b[k]), k


def test_bad_node_sets_device_check(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["tiny"]
    gtrie, _ = build_tries(wl, _catalog(wl))
    st = _init_state(1, wl.W, wl.T)
    st["node"][0, 0] = 10_000                                 # no such node at level 0
    ws = bd.workspace(bd.beam_select_workspace_size(1, wl.W, wl.K, wl.V))
    lg = synth.logits(wl, 0, device=DEV)
    res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K, ws=ws)
    assert bd.read_status(ws) == bd.ERR_DEVICE_CHECK
    assert int(res["n_live_out"][0]) == 0                       # the bad beam contributed nothing
    assert bd.read_status(ws) == 0                              # reading clears the word


# ---------------------------------------------------------------------------- Gumbel top-k

@pytest.mark.parametrize("temperature,seed", [(1.0, 1), (0.5, 2), (2.0, (1 << 40) + 3)])
def test_gumbel_tiny_chain_bitexact(gpu_lib, temperature, seed):
    """Temperature > 0: Gumbel top-k with the counter-based noise drawn on each
    side by its own Philox4x32-10 and float32 logarithm; selections, scores
    (noise-free), nodes and slot rows equal the oracle's bit for bit."""
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl, _catalog(wl), temperature=temperature, seed=seed)


def test_gumbel_tiny_open_vocab(gpu_lib):
    wl = synth.WORKLOADS["tiny"].scaled(levels=0, n_items=0)
    run_chain(wl, K=5, temperature=0.8, seed=11)


def test_gumbel_qwen06b_chain_bitexact(gpu_lib):
    wl = synth.WORKLOADS["qwen06b"]
    run_chain(wl, _catalog(wl), temperature=1.0, seed=20261202)


def test_gumbel_onerec17b_full_size_bitexact(gpu_lib):
    """The 4 x 512-beam shape with the noise (first two steps)."""
    wl = synth.WORKLOADS["onerec17b"]
    run_chain(wl, _catalog(wl), steps=2, temperature=0.7, seed=5)


def test_gumbel_production_path(gpu_lib):
    """Own log-sum-exp (the one-launch stream kernel) in Gumbel mode against the
    oracle's chain."""
    wl = synth.WORKLOADS["qwen06b"]
    assert run_chain_own_lse(wl, items=_catalog(wl), temperature=1.0, seed=99) >= 1


def test_gumbel_differs_from_deterministic_and_repeats(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"]
    gtrie, _ = build_tries(wl, _catalog(wl))
    st = _init_state(wl.R, wl.W, wl.T)
    lg = synth.logits(wl, 0, device=DEV)
    det = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K)
    g1 = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K,
                        temperature=1.0, seed=4)
    g2 = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K,
                        temperature=1.0, seed=4)
    assert not torch.equal(det["tokens"], g1["tokens"])
    for k in ("tokens", "parents", "cum_out", "node_out", "n_live_out", "slot_out"):
        assert torch.equal(g1[k], g2[k]), k


# ---------------------------------------------------------------------------- dense trie levels

def test_dense_masks_match_the_oracle_trie(gpu_lib):
    """Bit c of node n's mask is set exactly for the codes of n's children in
    the oracle's trie."""
    wl = synth.WORKLOADS["qwen06b"]
    gtrie, otr = build_tries(wl, _catalog(wl))
    for lv in (0, 1):
        assert gtrie.export_dense(lv) is None
        gtrie.make_dense(lv)
        m = gtrie.export_dense(lv).cpu().numpy().view(np.uint32)
        n_nodes = m.shape[0]
        for node in list(range(min(n_nodes, 300))) + [n_nodes - 1]:
            codes, _ = otr.children(lv, node)
            bits = np.zeros(m.shape[1] * 32, bool)
            bits[codes] = True
            got = ((m[node][:, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool).reshape(-1)
            assert np.array_equal(got, bits), (lv, node)
        gtrie.drop_dense(lv)
        assert gtrie.export_dense(lv) is None


def test_dense_tiny_chain_bitexact(gpu_lib):
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl, _catalog(wl), dense_levels=(0, 1, 2))


def test_dense_qwen06b_chain_bitexact(gpu_lib):
    wl = synth.WORKLOADS["qwen06b"]
    run_chain(wl, _catalog(wl), dense_levels=(0, 1))


def test_dense_onerec17b_bitexact_and_gumbel(gpu_lib):
    wl = synth.WORKLOADS["onerec17b"]
    items = _catalog(wl)
    run_chain(wl, items, steps=2, dense_levels=(0, 1))
    run_chain(wl, items, steps=2, dense_levels=(0, 1), temperature=0.9, seed=77)


def test_dense_masks_leave_the_one_launch_path_unchanged(gpu_lib):
    """With masks on levels 0 and 1 the one-launch path (no lse_in) still
    matches the oracle's chain: it enumerates the CSR lists."""
    wl = synth.WORKLOADS["qwen06b"]
    assert run_chain_own_lse(wl, items=_catalog(wl), dense_levels=(0, 1)) >= 1
