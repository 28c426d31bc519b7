"""The seeded input generators (`synth`): the recipe stated for the
workloads, and the properties the parity tests rely on (any few logits rows
regenerate alone; every tensor has its own stream)."""
import numpy as np
import torch

import synth


def test_logit_rows_regenerate_any_rows_alone():
    wl = synth.WORKLOADS["qwen06b"].scaled(W=70)
    full = synth.logits(wl, 1)
    assert full.shape == (1, 70, wl.V) and full.dtype == torch.float32
    for b0, b1 in ((0, 1), (60, 70), (63, 65), (5, 64)):
        assert torch.equal(synth.logit_rows(wl, 1, 0, b0, b1), full[0, b0:b1])
    # a wider beam draws the same first rows (blocks of 64 rows, one stream each)
    assert torch.equal(synth.logits(wl.scaled(W=130), 1)[:, :70], full)
    # another step or request is another stream
    assert not torch.equal(synth.logits(wl, 2), full)


def test_logit_distribution_and_spikes():
    wl = synth.WORKLOADS["fp8kv"].scaled(R=1, W=64)
    x = synth.logits(wl, 0).double()
    spikes = x > 6.0 * 3.0                        # N(0, 3) almost never passes 18; +8 spikes often do not,
    frac = ((x - synth.logits(wl.scaled(spike_p=0.0), 0).double()).abs() > 1e-6).double().mean().item()
    assert abs(frac - 0.01) < 0.001               # Bernoulli(0.01) spikes of +8
    assert spikes.double().mean().item() < 1e-4
    base = synth.logits(synth.WORKLOADS["qwen06b"].scaled(W=64), 0).double()
    assert abs(base.mean().item()) < 0.01 and abs(base.std().item() - 2.0) < 0.01   # N(0, 2)


def test_catalog_distinct_zipf_and_deterministic():
    wl = synth.WORKLOADS["qwen06b"].scaled(n_items=50_000)
    items = synth.catalog(wl)
    assert items.shape == (50_000, 3) and items.dtype == np.int32
    assert items.min() >= 0 and items.max() < wl.C
    assert len(np.unique(items, axis=0)) == len(items)
    assert np.array_equal(items, synth.catalog(wl))
    c0 = np.bincount(items[:, 0], minlength=wl.C)
    assert c0[0] > 20 * c0[wl.C // 2]            # Zipf(1.1): code 0 far above the median code
    tiny = synth.catalog(synth.WORKLOADS["tiny"])
    assert tiny.shape == (200, 3) and tiny.max() < 16


def test_prompt_lengths_and_offsets():
    wl = synth.WORKLOADS["fp8kv"]
    p = synth.prompt_lens(wl)
    assert p.shape == (4,) and p.min() >= 512 and p.max() <= 8192
    assert np.array_equal(p, synth.prompt_lens(wl))
    off = synth.prompt_offsets(wl)
    assert off[0] == 0 and np.array_equal(np.diff(off), p)


def test_attention_inputs_recipe():
    wl = synth.WORKLOADS["fp8kv"].scaled(R=2, prompt_lens=[100, 37], p_range=None, W=8, T=2)
    a = synth.attention_inputs(wl, 1)
    assert a["q"].dtype == torch.bfloat16 and a["q"].shape == (2, 8, 16, 128)
    assert a["shared_k"].dtype == torch.float8_e4m3fn and a["shared_k"].shape == (137, 8, 128)
    assert a["unshared_v"].shape == (2, 16, 8, 128)
    # per kv head scale = amax / 448 over the shared KV, and the largest code is the top of the range
    sk = a["shared_k"].float() * a["k_scale"].view(1, -1, 1)
    amax = sk.abs().amax(dim=(0, 2))
    assert torch.allclose(amax / synth.E4M3_MAX, a["k_scale"], rtol=0.07)
    assert a["shared_k"].float().abs().amax().item() == synth.E4M3_MAX
    # queries change with the step, the KV pools do not
    b = synth.attention_inputs(wl, 0)
    assert not torch.equal(a["q"], b["q"]) and torch.equal(a["shared_k"].view(torch.uint8),
                                                         b["shared_k"].view(torch.uint8))
