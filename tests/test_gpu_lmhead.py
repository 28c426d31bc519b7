"""LM head with the fused log-sum-exp against the oracle (float64 from the
same bf16 inputs), and the selection it feeds.

Tolerances: the GPU accumulates the bf16 products of each logit in float32
over hidden_dim terms; for logits of order 2 (weights scaled so) that is
below 1e-4 absolute, so the window logits are checked at 2e-4 and the row
log-sum-exp (a softmax-weighted mean of logit errors plus its own float32
folding) at 2e-4.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import lmhead as olm
from oracle import select as osel
from tests._helpers import build_tries

pytestmark = pytest.mark.gpu
DEV = "cuda"
ATOL_LOGIT = 2e-4
ATOL_LSE = 2e-4


def _inputs(rows, H, V, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    h = torch.randn(rows, H, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(V, H, generator=g, device=DEV) * (2.0 / H ** 0.5)).to(torch.bfloat16)   # logits ~ N(0, 2)
    return h, w


@pytest.mark.parametrize("rows,H,V,win", [(200, 256, 5000, (1000, 700)), (128, 64, 256, (0, 256)),
                                          (1, 128, 300, (299, 1)), (300, 512, 4097, (4000, 97))])
def test_lse_and_window_match_float64(gpu_lib, rows, H, V, win):
    from wide_beam_generative_gb300 import beamdec as bd
    h, w = _inputs(rows, H, V, rows + H)
    lse, lg = bd.beam_lmhead_lse(h, w, window_start=win[0], window_len=win[1])
    torch.cuda.synchronize()
    want_lse, want = olm.lse_rows(h.double().cpu().numpy(), w.double().cpu().numpy())
    assert np.abs(lse.cpu().numpy().astype(np.float64) - want_lse).max() < ATOL_LSE
    a, b = win[0], win[0] + win[1]
    got = lg[:, a:b].cpu().numpy().astype(np.float64)
    assert np.abs(got - want[:, a:b]).max() < ATOL_LOGIT


def test_full_size_sampled_rows(gpu_lib):
    """2048 rows x hidden 2048 x vocab 151936 (a 4 x 512-beam step of a
    Qwen3-1.7B-shaped head); 24 sampled rows checked against float64."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["onerec17b"]
    rows, H, V = wl.R * wl.W, 2048, wl.V
    h, w = _inputs(rows, H, V, 7)
    tb = int(wl.token_base()[2])
    lse, lg = bd.beam_lmhead_lse(h, w, window_start=tb, window_len=wl.C)
    torch.cuda.synchronize()
    pick = np.random.default_rng(0).choice(rows, 24, replace=False)
    want_lse, want = olm.lse_rows(h.double().cpu().numpy(), w.double().cpu().numpy(), rows=pick)
    assert np.abs(lse.cpu().numpy()[pick].astype(np.float64) - want_lse).max() < ATOL_LSE
    got = lg[pick, tb:tb + wl.C].cpu().numpy().astype(np.float64)
    assert np.abs(got - want[:, tb:tb + wl.C]).max() < ATOL_LOGIT


def test_selection_from_lmhead_window(gpu_lib):
    """qwen06b-shaped step 0 and 1 with logits from the fused LM head: the
    selection (lse_in from the head, children logits from the window) against
    the oracle's selection on float64 logits, allowing only near-cut trades."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"]
    R, W, K, V, H = wl.R, wl.W, wl.K, wl.V, 1024
    items = synth.catalog(wl)
    gtrie, otr = build_tries(wl, items)
    cum = torch.zeros((R, W), dtype=torch.float32, device=DEV)
    node = torch.zeros((R, W), dtype=torch.int32, device=DEV)
    n_live = torch.ones((R,), dtype=torch.int32, device=DEV)
    slot = torch.full((R, W, wl.T), -1, dtype=torch.int32, device=DEV)
    o_cum, o_node = np.zeros((R, W), np.float32), np.zeros((R, W), np.int64)
    o_nl, o_slot = np.ones(R, np.int32), np.full((R, W, wl.T), -1, np.int32)
    for t in range(2):
        h, w = _inputs(R * W, H, V, 100 + t)
        tb = int(wl.token_base()[t])
        lse, lg = bd.beam_lmhead_lse(h, w, window_start=tb, window_len=wl.C)
        res = bd.beam_select(lg.view(R, W, V), cum, node, n_live, slot, gtrie, t, t, K, lse_in=lse.view(R, W))
        lg64 = olm.logits64(h.double().cpu().numpy(), w.double().cpu().numpy()).reshape(R, W, V)
        ref = osel.beam_select(lg64.astype(np.float32), o_cum, o_node, o_nl, o_slot, otr, wl.token_base(),
                               t, t, W, K, lse32=np.array([[np.float32(osel.lse64(lg64[r, b])) for b in range(W)]
                                                          for r in range(R)]))
        n = int(ref["n_live_out"][0])
        assert int(res["n_live_out"][0]) == n
        g_s = res["cum_out"].cpu().numpy()[0, :n].astype(np.float64)
        o_s = ref["cum_out"][0, :n].astype(np.float64)
        assert np.abs(g_s - o_s).max() < 1e-3
        gp, gt = res["parents"].cpu().numpy()[0, :n], res["tokens"].cpu().numpy()[0, :n]
        if not (np.array_equal(gp, ref["parents"][0, :n]) and np.array_equal(gt, ref["tokens"][0, :n])):
            cut = o_s[-1]
            lookup = {(p, k): sc for p, k, sc in zip(ref["parents"][0, :n], ref["tokens"][0, :n], o_s)}
            for key in set(zip(gp, gt)) ^ set(lookup):
                if key in lookup:
                    assert abs(lookup[key] - cut) < 1e-3
            break
        cum, node, n_live, slot = res["cum_out"], res["node_out"], res["n_live_out"], res["slot_out"]
        o_cum, o_node, o_nl, o_slot = ref["cum_out"], ref["node_out"], ref["n_live_out"], ref["slot_out"]


def test_mbarrier_timeout_is_reported(gpu_lib):
    """A bounded mbarrier wait that runs out ends the launch with
    BEAMDEC_ERR_TIMEOUT instead of hanging: the workspace's probe hook makes
    every CTA wait 1000 polls on a barrier nothing completes before it issues
    any copy or MMA (a flag that nothing sets).  With the hook cleared the
    same workspace gives the float64 result."""
    from wide_beam_generative_gb300 import beamdec as bd
    rows, H, V = 200, 256, 5000
    h, w = _inputs(rows, H, V, 11)
    ws = bd.workspace(bd.beam_lmhead_workspace_size(rows, V))
    hooks = ws[:24].view(torch.int32)
    hooks[5] = 1000          # probe_polls
    bd.beam_lmhead_lse(h, w, ws=ws)
    assert bd.read_status(ws) == bd.ERR_TIMEOUT
    hooks[5] = 0
    lse, _ = bd.beam_lmhead_lse(h, w, ws=ws)
    assert bd.read_status(ws) == 0
    want_lse, _ = olm.lse_rows(h.double().cpu().numpy(), w.double().cpu().numpy())
    assert np.abs(lse.cpu().numpy().astype(np.float64) - want_lse).max() < ATOL_LSE
