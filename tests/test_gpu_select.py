"""GPU parity of beam_trie_build and beam_select against the CPU oracle.

Selection is compared bit for bit (tokens, parents, scores, child nodes, slot
rows, live counts) when both sides score against the same float32
log-sum-exp: the oracle's float64 value rounded to float32.  Two kernels take
it: the expansion kernel through ``lse_in`` (mode "expand"), and the
one-launch stream kernel that every benchmark number comes from, through
``score_lse`` (mode "stream": the kernel still streams every row for its own
normaliser, which is checked against float64 within 1e-5 at every step).
The production call (the kernel scores against its own normaliser) is
compared with the oracle at every step from the oracle's state: bit for bit
where the two normalisers' roundings trade no candidate, otherwise every
selected candidate is checked for validity and every difference for a score
at the cut.
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
              seed=0, dense_levels=(), mode="expand"):
    """Decode `steps` steps on the GPU and in the oracle in lockstep
    (temperature > 0: Gumbel top-k under `seed` on both sides).  Both sides
    score against the oracle's float32 normaliser: passed as ``lse_in``
    (mode "expand": the expansion kernel) or as ``score_lse`` (mode
    "stream": the one-launch kernel, whose own log-sum-exp must then lie
    within 1e-5 of float64)."""
    from wide_beam_generative_gb300 import beamdec as bd
    assert mode in ("expand", "stream")
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
        norm = torch.from_numpy(np.nan_to_num(lse32)).to(DEV)
        res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, t, t, K,
                             lse_in=norm if mode == "expand" else None,
                             score_lse=norm if mode == "stream" else None, ws=ws,
                             temperature=temperature, seed=seed)
        ref = osel.beam_select(lg_np, o_cum, o_node, o_nl, o_slot, otr, wl.token_base(), t, t, W, K,
                               lse32=lse32, temperature=temperature, seed=seed)
        if check:
            compare_select(res, ref, t, f"{wl.name} step {t} ({mode})")
            if mode == "stream":
                got = res["lse_out"].cpu().numpy()
                for r in range(wl.R):
                    n = int(o_nl[r])
                    assert np.abs(got[r, :n].astype(np.float64) - ref["lse64"][r, :n]).max() < ATOL_LSE
        assert bd.read_status(ws) == 0
        outs.append((res, ref))
        st = dict(cum=res["cum_out"], node=res["node_out"], n_live=res["n_live_out"], slot=res["slot_out"])
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]
    return outs


MODES = ["expand", "stream"]


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

@pytest.mark.parametrize("mode", MODES)
def test_tiny_chain_bitexact(gpu_lib, mode):
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl, _catalog(wl), mode=mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [1, 3, 8, 20])
@pytest.mark.parametrize("W", [1, 8, 37])
def test_tiny_chain_widths(gpu_lib, K, W, mode):
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl.scaled(W=W), _catalog(wl), K=K, W=W, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_tiny_open_vocab_with_ties(gpu_lib, mode):
    wl = synth.WORKLOADS["tiny"].scaled(name="tiny-open", levels=0, n_items=0, W=16)

    def quantised(t):   # integer logits: many exact ties in score
        return torch.round(synth.logits(wl, t, device=DEV))
    run_chain(wl, None, K=5, W=16, logit_fn=quantised, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_constant_logits_all_ties(gpu_lib, mode):
    wl = synth.WORKLOADS["tiny"].scaled(name="tiny-const", levels=0, n_items=0, W=12)
    run_chain(wl, None, K=7, W=12, logit_fn=lambda t: torch.zeros((1, 12, wl.V), device=DEV), mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_qwen06b_chain_bitexact(gpu_lib, mode):
    wl = synth.WORKLOADS["qwen06b"]
    run_chain(wl, _catalog(wl), mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_open_vocab_large_vocab(gpu_lib, mode):
    wl = synth.WORKLOADS["openvocab"].scaled(W=48, K=48, T=4)
    run_chain(wl, None, steps=3, mode=mode)
    run_chain(wl, None, steps=2, K=5, mode=mode)          # top_k < beam_width: per-beam cap binds


@pytest.mark.parametrize("mode", MODES)
def test_large_rows_with_ties(gpu_lib, mode):
    """Rows of 151936 candidates (more than the key cache holds) with
    whole-number logits, so exact score ties surround the top_k-th key, with
    top_k below and above beam_width; and constant rows of 20000, where every
    key ties (one bin holds them all: the radix fallback)."""
    wl = synth.WORKLOADS["openvocab"].scaled(name="ov-ties", R=2, W=64, K=64, T=3)

    def whole(t):
        return torch.round(synth.logits(wl, t, device=DEV))
    run_chain(wl, None, steps=3, logit_fn=whole, mode=mode)
    run_chain(wl, None, steps=2, K=700, logit_fn=whole, mode=mode)
    run_chain(wl, None, steps=2, K=9, logit_fn=whole, mode=mode)
    wc = synth.WORKLOADS["openvocab"].scaled(name="ov-const", R=1, W=16, K=16, T=2, V=20000)
    run_chain(wc, None, steps=2, logit_fn=lambda t: torch.full((1, 16, 20000), 1.5, device=DEV), mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_open_vocab_odd_vocab(gpu_lib, mode):
    """An odd vocabulary above the key cache (12289 tokens): every row but
    the first starts off a 16-byte boundary, so the normaliser stream, the
    cut seeds and the wide-row select take their unaligned paths; few live
    beams at step 0, then a top_k of 3 and of 2000."""
    wl = synth.WORKLOADS["openvocab"].scaled(name="ov-odd", R=2, W=24, K=24, T=4, V=12289)
    run_chain(wl, None, steps=3, mode=mode)
    run_chain(wl, None, steps=2, K=3, mode=mode)
    run_chain(wl, None, steps=2, K=2000, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_trie_node_above_key_cache(gpu_lib, mode):
    """A root with 16384 children (more than the 8192 keys a block caches):
    the large-row path enumerates the node's CSR code list."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="wide-root", levels=2, C=16384, n_items=120_000, zipf=None,
                                           W=32, K=32, T=2)
    items = _catalog(wl)
    run_chain(wl, items, mode=mode)
    run_chain(wl, items, K=3000, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_gumbel_large_rows(gpu_lib, mode):
    """Gumbel top-k over the whole 151936-token vocabulary (ordering keys
    with noise through the large-row path)."""
    wl = synth.WORKLOADS["openvocab"].scaled(name="ov-gumbel", R=1, W=40, K=40, T=2)
    run_chain(wl, None, steps=2, temperature=0.9, seed=31, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_onerec17b_full_size_bitexact(gpu_lib, mode):
    """The benchmarked workload at full size: 4 requests x 512 beams, top_k 512,
    4M-item Zipf catalog, vocab 151936, all three steps (the third is the
    step the benchmark times, on the kernel it times in mode "stream")."""
    wl = synth.WORKLOADS["onerec17b"]
    outs = run_chain(wl, _catalog(wl), mode=mode)
    assert int(outs[-1][0]["n_live_out"].min()) == wl.W


@pytest.mark.parametrize("mode", MODES)
def test_fp8kv_full_size_bitexact(gpu_lib, mode):
    """4 requests x 1000 beams, top_k 128 < W, 4 SID levels of 4096, 2M items,
    logits N(0,3) with 1% spikes of +8, all four steps."""
    wl = synth.WORKLOADS["fp8kv"]
    run_chain(wl, _catalog(wl), mode=mode)


def check_open_vocab_topw(res, cum_in, n_live_in, lg, lse32, slot_in, step, W, K):
    """Exact check of an open-vocabulary selection with top_k >= W, with no
    full sort: with top_k >= W the selection is the top-W of every (beam,
    token) pair of the live rows, so it is exactly right when (1) every
    selected score equals its recomputation fl32(cum + fl32(logit - lse)),
    (2) the pairs are unique and strictly ordered by (score desc, beam asc,
    token asc), and (3) exactly n_live' candidates of the whole grid lie at or
    before the last selected one in that order.  Also the live count, the dead
    rows, the child nodes (-1 without a trie) and the slot rows."""
    assert K >= W
    R, V = lg.shape[0], lg.shape[2]
    for r in range(R):
        n_in = int(n_live_in[r])
        nl = int(res["n_live_out"][r])
        assert nl == min(W, n_in * min(K, V))
        par = res["parents"][r, :nl].long()
        tok = res["tokens"][r, :nl].long()
        assert bool((par >= 0).all() and (par < n_in).all() and (tok >= 0).all() and (tok < V).all())
        assert torch.unique(par * V + tok).numel() == nl                       # (2) unique
        s = cum_in[r, par] + (lg[r, par, tok] - lse32[r, par])
        assert torch.equal(s, res["cum_out"][r, :nl])                         # (1)
        before = (s[:-1] > s[1:]) | ((s[:-1] == s[1:]) & ((par[:-1] < par[1:]) |
                                                          ((par[:-1] == par[1:]) & (tok[:-1] < tok[1:]))))
        assert bool(before.all())                                             # (2) order
        sW, bW, tW = s[-1], int(par[-1]), int(tok[-1])
        count = 0
        for b0 in range(0, n_in, 500):
            b1 = min(n_in, b0 + 500)
            sc = cum_in[r, b0:b1, None] + (lg[r, b0:b1] - lse32[r, b0:b1, None])
            bidx = torch.arange(b0, b1, device=DEV)[:, None]
            tidx = torch.arange(V, device=DEV)[None, :]
            better = (sc > sW) | ((sc == sW) & ((bidx < bW) | ((bidx == bW) & (tidx <= tW))))
            count += int(better.sum())
        assert count == nl                                                    # (3)
        assert bool((res["tokens"][r, nl:] == -1).all() and (res["parents"][r, nl:] == -1).all())
        assert bool(torch.isneginf(res["cum_out"][r, nl:]).all())
        assert bool((res["node_out"][r] == -1).all())
        so = res["slot_out"][r]
        assert torch.equal(so[:nl, :step], slot_in[r, par, :step])
        assert torch.equal(so[:nl, step], step * W + torch.arange(nl, device=DEV, dtype=torch.int32))
        assert bool((so[:nl, step + 1:] == -1).all() and (so[nl:] == -1).all())


@pytest.mark.parametrize("mode", MODES)
def test_openvocab_full_size(gpu_lib, mode):
    """2 requests x 5000 beams, top_k 5000, open vocabulary 151936: 25M-candidate
    pools (the cooperative global-selection kernel).  Step 0 is compared with
    the oracle bit for bit; steps 1-3 are checked exactly by counting
    (check_open_vocab_topw), each from the previous step's state, against the
    float64 normaliser rounded to float32 (torch's float64 log-sum-exp)."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["openvocab"]
    outs = run_chain(wl, None, steps=1, mode=mode)
    res0 = outs[0][0]
    st = dict(cum=res0["cum_out"], node=res0["node_out"], n_live=res0["n_live_out"], slot=res0["slot_out"])
    ws = bd.workspace(bd.beam_select_workspace_size(wl.R, wl.W, wl.K, wl.V))
    for t in (1, 2, 3):
        lg = synth.logits(wl, t, device=DEV)
        lse64 = torch.logsumexp(lg.double(), dim=-1)
        lse32 = lse64.float()
        res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, t, t, wl.K, ws=ws,
                             lse_in=lse32 if mode == "expand" else None,
                             score_lse=lse32 if mode == "stream" else None)
        assert bd.read_status(ws) == 0
        if mode == "stream":
            nl = st["n_live"].cpu().tolist()
            for r in range(wl.R):
                err = (res["lse_out"][r, :nl[r]].double() - lse64[r, :nl[r]]).abs().max()
                assert float(err) < ATOL_LSE
        check_open_vocab_topw(res, st["cum"], st["n_live"].cpu().tolist(), lg, lse32, st["slot"], t, wl.W,
                              wl.K)
        st = dict(cum=res["cum_out"], node=res["node_out"], n_live=res["n_live_out"], slot=res["slot_out"])
        del lg, lse64


# ---------------------------------------------------------------------------- full path

def run_chain_own_lse(wl, steps=None, items=None, temperature=0.0, seed=0, dense_levels=()):
    """The production call (the one-launch kernel scores the candidates
    against its own normaliser) against the oracle's own float64 chain, at
    every step.  Each step starts both sides from the oracle's state (copied
    to the device), so every step is compared whatever happened before.

    Per step: the kernel's log-sum-exp within 1e-5 of float64; live counts
    equal; every GPU-selected candidate valid: a live parent, a unique
    (parent, token) pair, a token among the children of the parent's trie
    node with the matching child node (any token and node -1 without a
    trie), the slot row of the parent followed by step*W + j, a score within
    2e-5 of the oracle's score of that candidate; and the GPU's list in
    non-increasing score order with equal scores by (parent, token).  Where the
    (parent, token) lists are equal, child nodes and slot rows are equal too.
    Where they differ, the two normalisers' independent float32 roundings
    traded near-ties: every candidate in only one list scores within 4e-5 of
    the cut, and the GPU's order inverts no pair whose oracle scores differ by
    4e-5 or more.  Returns the number of steps at which every request's
    list equalled the oracle's."""
    from wide_beam_generative_gb300 import beamdec as bd
    W, K, R, T = wl.W, wl.K, wl.R, wl.T
    steps = T if steps is None else steps
    gtrie, otr = build_tries(wl, items) if wl.levels else (None, None)
    for lv in dense_levels:
        gtrie.make_dense(lv)
    tb = wl.token_base()
    o_cum = np.zeros((R, W), np.float32)
    o_node = np.zeros((R, W), np.int64)
    o_nl = np.ones(R, np.int32)
    o_slot = np.full((R, W, T), -1, np.int32)
    ws = bd.workspace(bd.beam_select_workspace_size(R, W, K, wl.V))
    exact = 0
    for t in range(steps):
        lg = synth.logits(wl, t, device=DEV)
        lg_np = lg.cpu().numpy()
        st = dict(cum=torch.from_numpy(o_cum).to(DEV), node=torch.from_numpy(o_node.astype(np.int32)).to(DEV),
                  n_live=torch.from_numpy(o_nl).to(DEV), slot=torch.from_numpy(o_slot).to(DEV))
        res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, t, t, K, ws=ws,
                             temperature=temperature, seed=seed)
        assert bd.read_status(ws) == 0
        ref = osel.beam_select(lg_np, o_cum, o_node, o_nl, o_slot, otr, tb, t, t,
                               W, K, temperature=temperature, seed=seed)
        got_lse = res["lse_out"].cpu().numpy()
        g = {k: res[k].cpu().numpy() for k in ("parents", "tokens", "cum_out", "node_out", "n_live_out",
                                               "slot_out")}
        all_same = True
        for r in range(R):
            nl_in = int(o_nl[r])
            assert np.abs(got_lse[r, :nl_in].astype(np.float64) - ref["lse64"][r, :nl_in]).max() < ATOL_LSE
            n = int(ref["n_live_out"][r])
            assert int(g["n_live_out"][r]) == n
            gp, gt, gs = g["parents"][r, :n], g["tokens"][r, :n], g["cum_out"][r, :n].astype(np.float64)
            # ---- validity of every GPU-selected candidate
            assert np.all((gp >= 0) & (gp < nl_in))
            assert len(set(zip(gp.tolist(), gt.tolist()))) == n
            for j in range(n):
                p, v = int(gp[j]), int(gt[j])
                if otr is not None:
                    codes, kids = otr.children(t, int(o_node[r, p]))
                    hit = np.nonzero(codes == v - int(tb[t]))[0]
                    assert len(hit) == 1, (r, j, p, v)
                    assert int(g["node_out"][r, j]) == int(kids[hit[0]])
                else:
                    assert 0 <= v < wl.V and int(g["node_out"][r, j]) == -1
                s_o = osel.candidate_scores(lg_np[r, p, v], o_cum[r, p], np.float32(ref["lse64"][r, p]))
                assert abs(float(s_o) - gs[j]) < 2e-5
            assert np.array_equal(g["slot_out"][r, :n, :t], o_slot[r, gp, :t])
            assert np.array_equal(g["slot_out"][r, :n, t], t * W + np.arange(n))
            if temperature == 0:
                ok = (gs[:-1] > gs[1:]) | ((gs[:-1] == gs[1:]) & ((gp[:-1] < gp[1:]) |
                                                                   ((gp[:-1] == gp[1:]) & (gt[:-1] < gt[1:]))))
                assert np.all(ok)
            # ---- against the oracle's list
            o_s = ref["cum_out"][r, :n].astype(np.float64)
            assert np.abs(gs - o_s).max() < 2e-5
            if np.array_equal(gp, ref["parents"][r, :n]) and np.array_equal(gt, ref["tokens"][r, :n]):
                assert np.array_equal(g["node_out"][r, :n], ref["node_out"][r, :n])
                assert np.array_equal(g["slot_out"][r, :n, :t + 1], ref["slot_out"][r, :n, :t + 1])
                continue
            all_same = False
            cut = o_s[-1]
            g_set = set(zip(gp.tolist(), gt.tolist()))
            o_set = set(zip(ref["parents"][r, :n].tolist(), ref["tokens"][r, :n].tolist()))
            lookup = {(p, tk): sc for p, tk, sc in zip(ref["parents"][r, :n].tolist(),
                                                       ref["tokens"][r, :n].tolist(), o_s)}
            g_lookup = {(p, tk): sc for p, tk, sc in zip(gp.tolist(), gt.tolist(), gs)}
            for key in o_set - g_set:
                assert abs(lookup[key] - cut) < 4e-5
            for key in g_set - o_set:
                assert abs(g_lookup[key] - cut) < 6e-5
            o_score = np.array([lookup.get(key, g_lookup[key]) for key in zip(gp.tolist(), gt.tolist())])
            assert np.all(np.minimum.accumulate(o_score)[:-1] >= o_score[1:] - 4e-5)
        exact += int(all_same)
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]
    return exact


def test_full_path_own_lse(gpu_lib):
    """qwen06b, 3 steps, the one-launch selection against the oracle's chain."""
    wl = synth.WORKLOADS["qwen06b"]
    run_chain_own_lse(wl, items=_catalog(wl))


def test_onerec17b_full_size_own_lse(gpu_lib):
    """The benchmarked shape (4 x 512 beams, top_k 512) on the production path:
    row expansion in each row's last stream block and the request tail in the
    request's last row, against the oracle's chain."""
    wl = synth.WORKLOADS["onerec17b"]
    run_chain_own_lse(wl, items=_catalog(wl))


def test_fp8kv_full_size_own_lse(gpu_lib):
    """4 x 1000 beams, top_k 128, four SID levels: more than 1024 candidates at
    or above the cut's bin, so the tail takes the radix-narrowing path."""
    wl = synth.WORKLOADS["fp8kv"]
    run_chain_own_lse(wl, items=_catalog(wl))


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


def test_grid_barrier_timeout_is_reported(gpu_lib):
    """A bounded device wait that runs out ends the launch with
    BEAMDEC_ERR_TIMEOUT instead of hanging.  The workspace's test hooks ask
    the grid barrier for one arrival that no block supplies (a flag nothing
    sets) and cut its poll count to 1000, on a shape that takes the
    cooperative global-selection kernel (W > 4096); open vocabulary at step 0
    keeps every output index in range whatever the unsynchronised blocks
    read.  With the hooks cleared the same workspace selects correctly."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["tiny"].scaled(name="tiny-coop", levels=0, n_items=0, W=4100, K=2, T=1)
    R, W, V = 1, wl.W, wl.V
    ws = bd.workspace(bd.beam_select_workspace_size(R, W, wl.K, V))
    st = _init_state(R, W, 1)
    lg = synth.logits(wl, 0, rows=W, device=DEV)
    hooks = ws[:20].view(torch.int32)
    hooks[3] = 1000          # poll_limit
    hooks[4] = 1             # bar_extra
    bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, 0, wl.K, ws=ws)
    assert bd.read_status(ws) == bd.ERR_TIMEOUT
    hooks[3] = 0
    hooks[4] = 0
    res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], None, 0, 0, wl.K, ws=ws)
    assert bd.read_status(ws) == 0
    lg_np = lg.cpu().numpy()
    ref = osel.beam_select(lg_np, np.zeros((R, W), np.float32), np.zeros((R, W), np.int64),
                           np.ones(R, np.int32), np.full((R, W, 1), -1, np.int32), None, wl.token_base(),
                           0, 0, W, wl.K, lse32=oracle_lse32(lg_np, np.ones(R, np.int32)))
    assert int(res["n_live_out"][0]) == 2
    assert res["tokens"][0, :2].cpu().tolist() == ref["tokens"][0, :2].tolist()
    assert res["parents"][0, :2].cpu().tolist() == [0, 0]


# ---------------------------------------------------------------------------- Gumbel top-k

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("temperature,seed", [(1.0, 1), (0.5, 2), (2.0, (1 << 40) + 3)])
def test_gumbel_tiny_chain_bitexact(gpu_lib, temperature, seed, mode):
    """Temperature > 0: Gumbel top-k with the counter-based noise drawn on each
    side by its own Philox4x32-10 and float32 logarithm; selections, scores
    (noise-free), nodes and slot rows equal the oracle's bit for bit."""
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl, _catalog(wl), temperature=temperature, seed=seed, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_gumbel_tiny_open_vocab(gpu_lib, mode):
    wl = synth.WORKLOADS["tiny"].scaled(levels=0, n_items=0)
    run_chain(wl, K=5, temperature=0.8, seed=11, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_gumbel_qwen06b_chain_bitexact(gpu_lib, mode):
    wl = synth.WORKLOADS["qwen06b"]
    run_chain(wl, _catalog(wl), temperature=1.0, seed=20261202, mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_gumbel_onerec17b_full_size_bitexact(gpu_lib, mode):
    """The 4 x 512-beam shape with the noise (all three steps)."""
    wl = synth.WORKLOADS["onerec17b"]
    run_chain(wl, _catalog(wl), temperature=0.7, seed=5, mode=mode)


def test_gumbel_production_path(gpu_lib):
    """Own log-sum-exp (the one-launch stream kernel) in Gumbel mode against the
    oracle's chain."""
    wl = synth.WORKLOADS["qwen06b"]
    run_chain_own_lse(wl, items=_catalog(wl), temperature=1.0, seed=99)


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


@pytest.mark.parametrize("mode", MODES)
def test_dense_tiny_chain_bitexact(gpu_lib, mode):
    """With masks on every level the candidates come from the masks both
    with lse_in (the expansion kernel) and without it (the rows' normalisers
    streamed first, then the same expansion); both equal the oracle."""
    wl = synth.WORKLOADS["tiny"]
    run_chain(wl, _catalog(wl), dense_levels=(0, 1, 2), mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_dense_qwen06b_chain_bitexact(gpu_lib, mode):
    wl = synth.WORKLOADS["qwen06b"]
    run_chain(wl, _catalog(wl), dense_levels=(0, 1), mode=mode)


@pytest.mark.parametrize("mode", MODES)
def test_dense_onerec17b_bitexact_and_gumbel(gpu_lib, mode):
    wl = synth.WORKLOADS["onerec17b"]
    items = _catalog(wl)
    run_chain(wl, items, steps=2, dense_levels=(0, 1), mode=mode)
    run_chain(wl, items, steps=2, dense_levels=(0, 1), temperature=0.9, seed=77, mode=mode)


def test_dense_masks_on_the_production_call(gpu_lib):
    """With masks on levels 0 and 1 the production call (no lse_in) streams
    the rows' normalisers and expands them from the masks (the expansion
    kernel runs; without masks it does not), and matches the oracle's chain
    at every step from the oracle's state."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"]
    items = _catalog(wl)
    run_chain_own_lse(wl, items=items, dense_levels=(0, 1))
    gtrie = bd.beam_trie_build(items, [wl.C] * wl.levels, wl.token_base(), wl.V)
    lg = synth.logits(wl, 0, device=DEV)
    st = _init_state(wl.R, wl.W, wl.T)
    counts = {}
    for masks in (False, True):
        if masks:
            gtrie.make_dense(0)
        bd.profile_enable(True)
        bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], gtrie, 0, 0, wl.K)
        torch.cuda.synchronize()
        counts[masks] = bd.profile_read()["bd_expand_kernel"][1]
        bd.profile_enable(False)
    assert counts == {False: 0, True: 1}
