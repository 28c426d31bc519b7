"""Pins for the oracle's beam attention and KV decoding (CPU only)."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import attention as oatt
from oracle import dequant
from tests.golden import read_kv


def _raw(t: torch.Tensor):
    """Raw storage of a tensor as numpy (float32 / uint16 bf16 bits / uint8 e4m3 bits)."""
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def make_inp(wl, step=0):
    a = synth.attention_inputs(wl, step)
    return dict(q=_raw(a["q"]), shared_k=_raw(a["shared_k"]), shared_v=_raw(a["shared_v"]),
                unshared_k=_raw(a["unshared_k"]), unshared_v=_raw(a["unshared_v"]),
                k_scale=a["k_scale"].numpy(), v_scale=a["v_scale"].numpy(),
                prompt_offsets=a["prompt_offsets"].numpy(), q_dtype=wl.q_dtype,
                kv_dtype=wl.kv_dtype)


def _rand_slots(wl, step, seed=0):
    rng = np.random.default_rng(seed)
    slot = np.full((wl.R, wl.W, wl.T), -1, np.int32)
    for t in range(step + 1):
        slot[:, :, t] = t * wl.W + rng.integers(0, wl.W, size=(wl.R, wl.W))
    return slot


def test_e4m3_and_bf16_decoding_match_torch():
    bits = np.arange(256, dtype=np.uint8)
    ours = dequant.e4m3_bits_to_f64(bits)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).float().double().numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), ~finite)
    assert np.array_equal(ours[finite], ref[finite])
    assert ours[0x38] == 1.0 and ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9
    b16 = np.random.default_rng(0).integers(0, 65536, 4096).astype(np.uint16)
    b16 = b16[(b16 & 0x7F80) != 0x7F80]                          # finite patterns
    ref16 = torch.from_numpy(b16.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(dequant.bf16_bits_to_f64(b16), ref16)


def test_golden_two_keys():
    g = read_kv("attn_small.txt")
    inp = dict(q=np.array(g["q"], np.float32).reshape(1, 1, 1, 2),
               shared_k=np.array(g["k0"], np.float32).reshape(1, 1, 2),
               shared_v=np.array(g["v0"], np.float32).reshape(1, 1, 2),
               unshared_k=np.array(g["k1"], np.float32).reshape(1, 1, 1, 2),
               unshared_v=np.array(g["v1"], np.float32).reshape(1, 1, 1, 2),
               prompt_offsets=np.array([0, 1]), q_dtype=0, kv_dtype=0)
    o = oatt.attention_decode(inp, np.zeros((1, 1, 1), np.int32), np.array([1]), 0)
    np.testing.assert_allclose(o[0, 0, 0], g["o"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("name", ["tiny"])
@pytest.mark.parametrize("step", [0, 2])
def test_split_equals_unsplit(name, step):
    wl = synth.WORKLOADS[name]
    inp = make_inp(wl, step)
    slot = _rand_slots(wl, step)
    n_live = np.array([wl.W - 2])
    a = oatt.attention_decode(inp, slot, n_live, step)
    b = oatt.attention_split(inp, slot, n_live, step, chunk=48)
    assert np.abs(a - b).max() < 1e-12
    assert np.all(a[:, wl.W - 2:] == 0)                       # dead rows are zero


def test_bf16_and_e4m3_split_equals_unsplit():
    for kvd in (synth.BF16, synth.E4M3):
        wl = synth.WORKLOADS["tiny"].scaled(name="tiny-q", Hq=4, Hkv=2, q_dtype=synth.BF16,
                                            kv_dtype=kvd, prompt_lens=[40, 17], R=2)
        inp = make_inp(wl, 1)
        slot = _rand_slots(wl, 1)
        n = np.array([wl.W, 3])
        a = oatt.attention_decode(inp, slot, n, 1)
        b = oatt.attention_split(inp, slot, n, 1, chunk=16)
        assert np.abs(a - b).max() < 1e-12


def _bruteforce_one(q, keys, vals, scale):
    s = [scale * sum(qi * ki for qi, ki in zip(q, k)) for k in keys]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = sum(e)
    return [sum(e[i] * vals[i][c] for i in range(len(keys))) / z for c in range(len(q))]


def test_pure_python_bruteforce():
    wl = synth.WORKLOADS["tiny"].scaled(name="tiny-bf", prompt_lens=[12], d=8, W=3)
    inp = make_inp(wl, 2)
    slot = _rand_slots(wl, 2, seed=5)
    o = oatt.attention_decode(inp, slot, np.array([3]), 2)
    q = inp["q"].astype(np.float64)
    for j in range(3):
        for h in range(2):
            keys = [inp["shared_k"][i, 0].tolist() for i in range(12)] + \
                   [inp["unshared_k"][0, s, 0].tolist() for s in slot[0, j, :3]]
            vals = [inp["shared_v"][i, 0].tolist() for i in range(12)] + \
                   [inp["unshared_v"][0, s, 0].tolist() for s in slot[0, j, :3]]
            want = _bruteforce_one(q[0, j, h].tolist(), keys, vals, 1 / math.sqrt(8))
            assert np.abs(o[0, j, h] - np.array(want)).max() < 1e-12


def _one_head_case(P, L, d=4, seed=0):
    rng = np.random.default_rng(seed)
    return dict(q=rng.normal(size=(1, 2, 1, d)).astype(np.float32),
                shared_k=rng.normal(size=(P, 1, d)).astype(np.float32),
                shared_v=rng.normal(size=(P, 1, d)).astype(np.float32),
                unshared_k=rng.normal(size=(1, 2 * L, 1, d)).astype(np.float32),
                unshared_v=rng.normal(size=(1, 2 * L, 1, d)).astype(np.float32),
                prompt_offsets=np.array([0, P]), q_dtype=0, kv_dtype=0)


def test_special_cases():
    # one key (empty prompt, step 0): o = v
    inp = _one_head_case(0, 1)
    slot = np.array([[[0], [1]]], np.int32)
    o = oatt.attention_decode(inp, slot, np.array([2]), 0)
    assert np.allclose(o[0, 0, 0], inp["unshared_v"][0, 0, 0], atol=1e-15)
    assert np.allclose(o[0, 1, 0], inp["unshared_v"][0, 1, 0], atol=1e-15)
    # all keys equal: uniform softmax, o = mean of the values
    inp = _one_head_case(5, 2)
    inp["shared_k"][:] = 0.5
    inp["unshared_k"][:] = 0.5
    slot = np.array([[[0, 2], [1, 3]]], np.int32)
    o = oatt.attention_decode(inp, slot, np.array([2]), 1)
    vals = np.concatenate([inp["shared_v"][:, 0], inp["unshared_v"][0, [0, 2], 0]])
    assert np.allclose(o[0, 0, 0], vals.astype(np.float64).mean(0), atol=1e-14)
    # q = 0: uniform as well
    inp = _one_head_case(7, 2, seed=1)
    inp["q"][:] = 0
    o = oatt.attention_decode(inp, slot, np.array([2]), 1)
    vals = np.concatenate([inp["shared_v"][:, 0], inp["unshared_v"][0, [1, 3], 0]])
    assert np.allclose(o[0, 1, 0], vals.astype(np.float64).mean(0), atol=1e-14)
    # beams sharing one parent chain and one query give identical rows
    inp = _one_head_case(9, 2, seed=2)
    inp["q"][0, 1] = inp["q"][0, 0]
    slot = np.array([[[0, 2], [0, 2]]], np.int32)
    o = oatt.attention_decode(inp, slot, np.array([2]), 1)
    assert np.array_equal(o[0, 0], o[0, 1])
