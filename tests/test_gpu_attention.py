"""GPU parity of beam_attn_decode against the float64 oracle on the same
quantised inputs.  Tolerances (absolute): fp32 2e-5 (float32 accumulation of
O(1) terms over <= a few thousand keys), bf16 KV 1e-2, fp8 e4m3 KV 5e-2."""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from tests._helpers import ATOL_ATTN, oracle_attn_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _slots(wl, step, n_live, seed=0):
    g = torch.Generator().manual_seed(seed)
    slot = torch.full((wl.R, wl.W, wl.T), -1, dtype=torch.int32)
    for t in range(step + 1):
        slot[:, :, t] = t * wl.W + torch.randint(0, wl.W, (wl.R, wl.W), generator=g, dtype=torch.int32)
    return slot


def _run(wl, step, n_live, beams=None, seed=0):
    """Runs the library and the oracle on the same inputs."""
    from wide_beam_generative_gb300 import beamdec as bd
    a = synth.attention_inputs(wl, step, device=DEV)
    slot = _slots(wl, step, n_live, seed)
    nl = torch.tensor(n_live, dtype=torch.int32)
    maxp = int(synth.prompt_lens(wl).max())
    out = bd.beam_attn_decode(a["q"], a["shared_k"], a["shared_v"], a["prompt_offsets"], maxp,
                              a["unshared_k"], a["unshared_v"], slot.to(DEV), nl.to(DEV), step,
                              k_scale=a["k_scale"], v_scale=a["v_scale"])
    torch.cuda.synchronize()
    inp = oracle_attn_inputs(a, a["q"], wl)
    want = oatt.attention_decode(inp, slot.numpy(), nl.numpy(), step, beams=beams)
    got = out.double().cpu().numpy()
    return got, want, out


def _check(wl, got, want, beams=None, out_rounding=False):
    """Max abs error below the KV type's tolerance.  out_rounding: the bound
    also admits the bf16 output's own rounding of the expected value (at most
    2^-8 |want|), for outputs well above 1 (prompts of a few keys, where a
    row averages only a handful of values)."""
    tol = ATOL_ATTN[wl.kv_dtype]
    if beams is not None:
        got = np.stack([got[r, j] for r, j in beams])
        want = np.stack([want[r, j] for r, j in beams])
    excess = np.abs(got - want) - (2.0 ** -8 * np.abs(want) if out_rounding else 0.0)
    err = excess.max()
    assert err < tol, f"max abs error {err} >= {tol}"
    return err


@pytest.mark.parametrize("step", [0, 1, 2])
def test_tiny_fp32(gpu_lib, step):
    wl = synth.WORKLOADS["tiny"]
    got, want, _ = _run(wl, step, [wl.W - 3])
    _check(wl, got, want)
    assert np.all(got[:, wl.W - 3:] == 0)                     # dead rows are zeros


def test_qwen06b_bf16_full(gpu_lib):
    wl = synth.WORKLOADS["qwen06b"]
    got, want, _ = _run(wl, 2, [wl.W])
    _check(wl, got, want)


def test_ragged_prompts_and_tails(gpu_lib):
    """Prompts that are not multiples of any tile, an empty prompt, partial
    beam tiles, d = 64 with bf16 and e4m3."""
    for kvd in (synth.BF16, synth.E4M3):
        for d in (64, 128):
            wl = synth.WORKLOADS["qwen06b"].scaled(name="ragged", R=3, prompt_lens=[1, 0, 333], d=d,
                                                   W=19, T=3, kv_dtype=kvd)
            got, want, _ = _run(wl, 1, [19, 7, 1])
            _check(wl, got, want)


def _tile_beams(wl, n_live, extra=2, seed=0):
    """The first and last live beam of every 256-row CTA tile (128 / G * 2
    beams per tile) of every request, plus `extra` random live beams."""
    per = 256 // wl.G
    rng = np.random.default_rng(seed)
    beams = []
    for r, nl in enumerate(n_live):
        js = set()
        for j0 in range(0, nl, per):
            js.update((j0, min(nl, j0 + per) - 1))
        js.update(int(x) for x in rng.integers(0, nl, extra))
        beams += [(r, j) for j in sorted(js)]
    return beams


def test_onerec17b_full_size_sampled(gpu_lib):
    """The benchmarked shape: 4 requests x 512 beams x 16 heads, prompts
    4096; the first and last beam of every 256-row tile of every request."""
    wl = synth.WORKLOADS["onerec17b"]
    beams = _tile_beams(wl, [wl.W] * wl.R)
    got, want, _ = _run(wl, 2, [wl.W] * wl.R, beams=beams)
    _check(wl, got, want, beams)


def test_fp8kv_full_size_sampled(gpu_lib):
    """4 requests x 1000 beams, e4m3 KV, ragged prompts; every tile's first
    and last live beam; dead beams zero."""
    wl = synth.WORKLOADS["fp8kv"]
    n_live = [wl.W, wl.W, 999, 500]
    beams = _tile_beams(wl, n_live)
    got, want, _ = _run(wl, 3, n_live, beams=beams)
    _check(wl, got, want, beams)
    assert np.all(got[2, 999:] == 0) and np.all(got[3, 500:] == 0)


def test_openvocab_full_size_sampled(gpu_lib):
    """2 requests x 5000 beams, 32 unshared tokens per beam at the last step
    (the merge kernel); every tile's first and last beam."""
    wl = synth.WORKLOADS["openvocab"]
    beams = _tile_beams(wl, [wl.W] * wl.R)
    got, want, _ = _run(wl, 31, [wl.W] * wl.R, beams=beams)
    _check(wl, got, want, beams)


def test_deterministic(gpu_lib):
    wl = synth.WORKLOADS["qwen06b"]
    _, _, a = _run(wl, 1, [wl.W])
    _, _, b = _run(wl, 1, [wl.W])
    assert torch.equal(a, b)


def test_bad_slot_sets_device_check(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["tiny"]
    a = synth.attention_inputs(wl, 0, device=DEV)
    slot = _slots(wl, 1, [wl.W])
    slot[0, 3, 1] = 10_000                                     # outside the T*W pool
    ws = bd.workspace(bd.beam_attn_workspace_size(1, wl.W, wl.Hq, wl.Hkv, wl.d, 256, wl.kv_dtype))
    bd.beam_attn_decode(a["q"], a["shared_k"], a["shared_v"], a["prompt_offsets"], 256,
                        a["unshared_k"], a["unshared_v"], slot.to(DEV),
                        torch.tensor([wl.W], dtype=torch.int32, device=DEV), 1, ws=ws)
    assert bd.read_status(ws) == bd.ERR_DEVICE_CHECK


@pytest.mark.parametrize("G,W,plens", [(2, 70, [300, 129]), (1, 200, [128, 1000]), (4, 33, [77, 512]),
                                       (8, 16, [2049, 5]), (16, 8, [640, 641])])
def test_tensor_core_shapes(gpu_lib, G, W, plens):
    """bf16, d = 128: the tcgen05 shared stage, with query tiles that end
    mid-tile, prompts that end mid-chunk and several prompt splits."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="tc", R=len(plens), prompt_lens=plens, Hq=2 * G, Hkv=2,
                                           W=W, T=3)
    got, want, _ = _run(wl, 1, [W, max(1, W - 5)])
    _check(wl, got, want)



def test_many_requests_dead_beams(gpu_lib):
    """Eight requests, one prompt split, dead beams and a partial last tile."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="many", R=8, prompt_lens=[256] * 8, W=250, T=4)
    got, want, _ = _run(wl, 3, [250, 250, 249, 128, 127, 1, 250, 200])
    _check(wl, got, want)
    assert np.all(got[5, 1:] == 0) and np.all(got[3, 128:] == 0)


def _merge_launches(fn):
    from wide_beam_generative_gb300 import beamdec as bd
    bd.profile_enable(True)
    fn()
    torch.cuda.synchronize()
    bd.profile_enable(False)
    return bd.profile_read()["bd_attn_merge_kernel"][1]


def test_fused_merge_empty_prompt_and_dead_beams(gpu_lib):
    """One prompt split (prompts of at most 128 keys), so the unshared stage
    and the merge run in the tensor-core kernel's epilogue: an empty prompt
    (the unshared tokens alone), a partial last tile, and dead beams in live
    and in wholly dead tiles."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="fused", R=3, prompt_lens=[0, 100, 128], W=300, T=3)
    res = {}

    def run():
        res["v"] = _run(wl, 2, [300, 129, 1])
    assert _merge_launches(run) == 0
    got, want, _ = res["v"]
    _check(wl, got, want, out_rounding=True)       # the empty prompt's rows reach |out| = 3.7
    _check(wl, got[1:], want[1:])                  # prompts of 100 and 128 keys: the plain bound
    assert np.all(got[1, 129:] == 0) and np.all(got[2, 1:] == 0)


def test_split_prompt_keeps_the_merge_kernel(gpu_lib):
    """Several prompt splits: the partials go through the merge kernel."""
    wl = synth.WORKLOADS["qwen06b"]
    res = {}

    def run():
        res["v"] = _run(wl, 2, [wl.W])
    assert _merge_launches(run) == 1
    got, want, _ = res["v"]
    _check(wl, got, want)


def test_fused_merge_fp8_kv(gpu_lib):
    """e4m3 KV with one prompt split: the epilogue reads the unshared rows as
    fp8 (K scale in the softmax scale, V scale on the output) and no merge
    kernel runs; an empty prompt, a one-key prompt and dead beams included."""
    wl = synth.WORKLOADS["fp8kv"].scaled(name="fused8", R=3, prompt_lens=[0, 1, 128], p_range=None, W=60, T=4)
    res = {}

    def run():
        res["v"] = _run(wl, 3, [60, 33, 1])
    assert _merge_launches(run) == 0
    got, want, _ = res["v"]
    _check(wl, got, want, out_rounding=True)
    assert np.all(got[1, 33:] == 0) and np.all(got[2, 1:] == 0)


def test_workspace_reused_across_calls(gpu_lib):
    """Three calls on one workspace (bf16 and e4m3 KV, split and unsplit
    prompts) give identical outputs, equal to the oracle's."""
    from wide_beam_generative_gb300 import beamdec as bd
    for wl, n_live in ((synth.WORKLOADS["qwen06b"], [50]),
                       (synth.WORKLOADS["fp8kv"].scaled(name="reuse8", R=2, prompt_lens=[700, 90], p_range=None,
                                                        W=30), [30, 11])):
        a = synth.attention_inputs(wl, 1, device=DEV)
        slot = _slots(wl, 1, n_live).to(DEV)
        nl = torch.tensor(n_live, dtype=torch.int32, device=DEV)
        maxp = int(synth.prompt_lens(wl).max())
        ws = bd.workspace(bd.beam_attn_workspace_size(wl.R, wl.W, wl.Hq, wl.Hkv, wl.d, maxp, wl.kv_dtype))
        outs = [bd.beam_attn_decode(a["q"], a["shared_k"], a["shared_v"], a["prompt_offsets"], maxp,
                                    a["unshared_k"], a["unshared_v"], slot, nl, 1, k_scale=a["k_scale"],
                                    v_scale=a["v_scale"], ws=ws).clone()
                for _ in range(3)]
        assert bd.read_status(ws) == 0
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
        inp = oracle_attn_inputs(a, a["q"], wl)
        want = oatt.attention_decode(inp, slot.cpu().numpy(), nl.cpu().numpy(), 1)
        _check(wl, outs[2].double().cpu().numpy(), want, out_rounding=True)


def test_fused_merge_bad_slot_sets_device_check(gpu_lib):
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"].scaled(name="fused", R=1, prompt_lens=[128], W=64, T=3)
    a = synth.attention_inputs(wl, 1, device=DEV)
    slot = _slots(wl, 1, [wl.W])
    slot[0, 5, 1] = 10_000                                     # outside the T*W pool
    ws = bd.workspace(bd.beam_attn_workspace_size(1, wl.W, wl.Hq, wl.Hkv, wl.d, 128, wl.kv_dtype))
    bd.beam_attn_decode(a["q"], a["shared_k"], a["shared_v"], a["prompt_offsets"], 128,
                        a["unshared_k"], a["unshared_v"], slot.to(DEV),
                        torch.tensor([wl.W], dtype=torch.int32, device=DEV), 1, ws=ws)
    assert bd.read_status(ws) == bd.ERR_DEVICE_CHECK


@pytest.mark.parametrize("G,W,plens,merge", [(1, 300, [128, 77], 0), (4, 70, [100, 128], 0),
                                             (8, 33, [128, 1], 0), (16, 20, [64, 128], 0)])
def test_fused_merge_group_sizes(gpu_lib, G, W, plens, merge):
    """One prompt split: the epilogue merges at every supported GQA group
    size; partial tiles and a one-key prompt."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="fusedg", R=len(plens), prompt_lens=plens, Hq=2 * G, Hkv=2,
                                           W=W, T=3)
    res = {}

    def run():
        res["v"] = _run(wl, 2, [W, max(1, W - 7)])
    assert _merge_launches(run) == merge
    got, want, _ = res["v"]
    _check(wl, got, want, out_rounding=True)
    assert np.all(got[1, max(1, W - 7):] == 0)


@pytest.mark.parametrize("step,merge", [(0, 0), (4, 0), (5, 0), (6, 1), (32, 1)])
def test_fused_merge_token_limit(gpu_lib, step, merge):
    """Up to 6 unshared tokens per beam are merged in the epilogue; 7 and
    more (here up to 33) go through the merge kernel; both against the
    oracle, with dead beams."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="fusedl", R=2, prompt_lens=[100, 128], W=40, T=33)
    res = {}

    def run():
        res["v"] = _run(wl, step, [40, 23])
    assert _merge_launches(run) == merge
    got, want, _ = res["v"]
    _check(wl, got, want)
    assert np.all(got[1, 23:] == 0)


@pytest.mark.parametrize("step,merge", [(5, 0), (31, 1)])
def test_fused_merge_fp8_kv_long(gpu_lib, step, merge):
    """e4m3 KV, one prompt split: 6 unshared tokens per beam merged in the
    epilogue, 32 in the merge kernel."""
    wl = synth.WORKLOADS["fp8kv"].scaled(name="fused8l", R=2, prompt_lens=[96, 128], p_range=None, W=50, T=32)
    res = {}

    def run():
        res["v"] = _run(wl, step, [50, 17])
    assert _merge_launches(run) == merge
    got, want, _ = res["v"]
    _check(wl, got, want, out_rounding=True)
    assert np.all(got[1, 17:] == 0)


def test_all_prompts_empty(gpu_lib):
    """No prompt key in any request (max_prompt_len 0, no shared K/V): the
    output is the softmax over the beams' unshared tokens alone."""
    wl = synth.WORKLOADS["qwen06b"].scaled(name="noprompt", R=2, prompt_lens=[0, 0], W=24, T=3)
    from wide_beam_generative_gb300 import beamdec as bd
    a = synth.attention_inputs(wl, 2, device=DEV)
    slot = _slots(wl, 2, [24, 10])
    nl = torch.tensor([24, 10], dtype=torch.int32)
    out = bd.beam_attn_decode(a["q"], None, None, a["prompt_offsets"], 0, a["unshared_k"], a["unshared_v"],
                              slot.to(DEV), nl.to(DEV), 2)
    inp = oracle_attn_inputs(a, a["q"], wl)
    want = oatt.attention_decode(inp, slot.numpy(), nl.numpy(), 2)
    _check(wl, out.double().cpu().numpy(), want, out_rounding=True)
    assert np.all(out[1, 10:].float().cpu().numpy() == 0)


def test_mbarrier_timeout_is_reported(gpu_lib):
    """A bounded mbarrier wait that runs out ends the tensor-core launch with
    BEAMDEC_ERR_TIMEOUT instead of hanging: the workspace's probe hook makes
    every CTA wait 1000 polls on a barrier nothing completes before it issues
    any copy or MMA (a flag that nothing sets).  With the hook cleared the
    same workspace matches the oracle."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["qwen06b"].scaled(name="probe", R=2, prompt_lens=[100, 128], W=40, T=3)
    a = synth.attention_inputs(wl, 2, device=DEV)
    slot = _slots(wl, 2, [40, 40])
    nl = torch.tensor([40, 40], dtype=torch.int32)
    ws = bd.workspace(bd.beam_attn_workspace_size(wl.R, wl.W, wl.Hq, wl.Hkv, wl.d, 128, wl.kv_dtype))
    hooks = ws[:24].view(torch.int32)

    def run():
        return bd.beam_attn_decode(a["q"], a["shared_k"], a["shared_v"], a["prompt_offsets"], 128,
                                   a["unshared_k"], a["unshared_v"], slot.to(DEV), nl.to(DEV), 2, ws=ws)
    hooks[5] = 1000          # probe_polls
    run()
    assert bd.read_status(ws) == bd.ERR_TIMEOUT
    hooks[5] = 0
    out = run()
    assert bd.read_status(ws) == 0
    want = oatt.attention_decode(oracle_attn_inputs(a, a["q"], wl), slot.numpy(), nl.numpy(), 2)
    _check(wl, out.double().cpu().numpy(), want)


@pytest.mark.parametrize("prompts,step", [([100, 0, 128], 2), ([300, 0, 517], 2), ([2048], 3)])
def test_prepared_e4m3_equals_the_per_call_copy(gpu_lib, prompts, step):
    """e4m3 prompt K/V dequantised once (beam_attn_prepare_prompt) and read by
    prepared decode calls gives the same bits as the copy each plain call
    makes, for a prompt in one split (merge in the shared stage) and split
    prompts (merge kernel), at steps where the shared stage starts its main
    loop before waiting; the copy persists across calls, and a prepared call
    naming another prompt K/V is reported."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl = synth.WORKLOADS["fp8kv"].scaled(name="prep", R=len(prompts), prompt_lens=prompts, p_range=None,
                                         W=200, T=4)
    a = synth.attention_inputs(wl, step, device=DEV)
    slot = _slots(wl, step, None).to(DEV)
    nl = torch.tensor([wl.W] * (wl.R - 1) + [wl.W - 57], dtype=torch.int32, device=DEV)
    maxp = int(synth.prompt_lens(wl).max())
    size = bd.beam_attn_workspace_size(wl.R, wl.W, wl.Hq, wl.Hkv, wl.d, maxp, bd.E4M3)
    ws_plain, ws_prep = bd.workspace(size, DEV), bd.workspace(size, DEV)

    def call(ws, prepared, shared_k=None):
        return bd.beam_attn_decode(a["q"], a["shared_k"] if shared_k is None else shared_k, a["shared_v"],
                                   a["prompt_offsets"], maxp, a["unshared_k"], a["unshared_v"], slot, nl,
                                   step, k_scale=a["k_scale"], v_scale=a["v_scale"], ws=ws,
                                   prepared=prepared)
    ref = call(ws_plain, False)
    bd.beam_attn_prepare_prompt(a["shared_k"], a["shared_v"], a["prompt_offsets"], maxp, wl.W, wl.Hq, ws_prep)
    got1 = call(ws_prep, True).clone()
    got2 = call(ws_prep, True)
    torch.cuda.synchronize()
    assert bd.read_status(ws_plain) == 0 and bd.read_status(ws_prep) == 0
    assert torch.equal(got1, ref) and torch.equal(got2, ref)
    call(ws_prep, True, shared_k=a["shared_k"].clone())   # not the prompt K/V the copy is of
    torch.cuda.synchronize()
    assert bd.read_status(ws_prep) == bd.ERR_DEVICE_CHECK
