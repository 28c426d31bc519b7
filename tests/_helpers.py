"""Shared glue of the GPU parity tests (marshalling only, no method arithmetic
beyond what the oracle provides)."""
import numpy as np
import torch

import synth
from oracle import select as osel

ATOL_ATTN = {synth.F32: 2e-5, synth.BF16: 1e-2, synth.E4M3: 5e-2}
ATOL_LSE = 1e-5


def raw(t: torch.Tensor):
    """Raw storage of a tensor as numpy (float32 / uint16 bf16 bits / uint8 e4m3 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def oracle_attn_inputs(a: dict, q: torch.Tensor, wl):
    return dict(q=raw(q), shared_k=raw(a["shared_k"]), shared_v=raw(a["shared_v"]),
                unshared_k=raw(a["unshared_k"]), unshared_v=raw(a["unshared_v"]),
                k_scale=a["k_scale"].cpu().numpy(), v_scale=a["v_scale"].cpu().numpy(),
                prompt_offsets=a["prompt_offsets"].cpu().numpy(), q_dtype=wl.q_dtype,
                kv_dtype=wl.kv_dtype)


def oracle_lse32(logits_np, n_live):
    """float32 rounding of the oracle's float64 log-sum-exp for every live row."""
    R, W = logits_np.shape[0], logits_np.shape[1]
    out = np.full((R, W), np.nan, np.float32)
    for r in range(R):
        for b in range(int(n_live[r])):
            out[r, b] = np.float32(osel.lse64(logits_np[r, b]))
    return out


def compare_select(res, ref, step, what=""):
    """Bit-exact comparison of every defined output of one expansion step."""
    nl_gpu = res["n_live_out"].cpu().numpy()
    assert np.array_equal(nl_gpu, ref["n_live_out"]), f"{what} n_live {nl_gpu} vs {ref['n_live_out']}"
    R = nl_gpu.shape[0]
    for r in range(R):
        n = int(nl_gpu[r])
        for k in ("tokens", "parents", "cum_out", "node_out"):
            g = res[k].cpu().numpy()[r]
            o = ref[k][r]
            assert np.array_equal(g[:n], o[:n].astype(g.dtype)), \
                f"{what} r{r} {k} first diff at {np.nonzero(g[:n] != o[:n])[0][:5]}"
            if k == "cum_out":
                assert np.isneginf(g[n:]).all()
            else:
                assert (g[n:] == -1).all(), f"{what} {k} dead rows"
        so = res["slot_out"].cpu().numpy()[r]
        assert np.array_equal(so[:n, :step + 1], ref["slot_out"][r, :n, :step + 1]), f"{what} slots"
        assert (so[:n, step + 1:] == -1).all() and (so[n:] == -1).all()


def build_tries(wl, items):
    from oracle import trie as otrie
    from wide_beam_generative_gb300 import beamdec as bd
    gpu = bd.beam_trie_build(items, [wl.C] * wl.levels, wl.token_base(), wl.V)
    return gpu, otrie.build_trie(items, wl.C)
