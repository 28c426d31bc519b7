"""Seeded synthetic inputs for the wide-beam decode step.

This module only draws random numbers and lays them out; it holds none of
the decode step's arithmetic (no softmax, no selection, no trie logic).  Both
the CPU oracle (``oracle/``) and the CUDA path are fed from here, so the two
always see identical bytes.

Workload shapes follow the five workloads the wide-beam decode step is
measured on (generative recommendation with semantic-ID items):

* ``tiny``      1 request, prompt 256, 2 q / 1 kv heads, d 64, W 8, K 8, 3 steps,
                vocab 512 with SID tokens 0-47 (3 levels x 16 codes), 200 items.
* ``qwen06b``   1 request, prompt 2048, 16/8 heads, d 128, W 50, K 50, 3 steps,
                vocab 151936, SID 3 x 8192, 1M Zipf(1.1) items.
* ``onerec17b`` 4 requests, prompts 4096, 16/8 heads, d 128, W 512, K 512,
                3 steps, SID 3 x 8192, 4M Zipf(1.1) items.
* ``fp8kv``     4 requests, prompts U[512, 8192], e4m3 KV, W 1000, K 128,
                4 steps, SID 4 x 4096, 2M items, logits N(0,3) + 1% spikes of +8.
* ``openvocab`` 2 requests, prompt 1024, W 5000, K 5000, 32 steps, no trie.

Random streams: every tensor has its own stream id, combined with the seed
into a Philox key (numpy) or a generator seed (torch), so that changing one
tensor's shape never shifts another tensor's values.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np
import torch

# dtype codes shared by the harness (the library header defines the same
# numbers for its ABI; these are plain data-layout tags)
F32, BF16, E4M3 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", BF16: "bf16", E4M3: "e4m3"}
E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    R: int                      # requests
    prompt_lens: list           # P_r per request (or None -> drawn, see p_range)
    Hq: int
    Hkv: int
    d: int
    W: int                      # beam_width
    K: int                      # top_k
    T: int                      # decode steps
    V: int                      # vocab
    levels: int                 # SID levels (0 = open vocab)
    C: int                      # codes per level
    n_items: int                # catalog size
    zipf: float | None          # Zipf exponent per level, None = uniform codes
    logit_sigma: float
    spike_p: float = 0.0
    spike_val: float = 0.0
    q_dtype: int = BF16
    kv_dtype: int = BF16
    out_dtype: int = BF16
    p_range: tuple | None = None  # (lo, hi) inclusive, drawn per request
    seed: int = 0

    @property
    def G(self):
        return self.Hq // self.Hkv

    def token_base(self):
        """First vocab id of each SID level's contiguous code range."""
        if self.levels == 0:
            return np.zeros(0, dtype=np.int32)
        if self.name.startswith("tiny"):
            return (np.arange(self.levels) * self.C).astype(np.int32)
        top = self.V - self.levels * self.C
        return (top + np.arange(self.levels) * self.C).astype(np.int32)

    def scaled(self, **kw):
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", R=1, prompt_lens=[256], Hq=2, Hkv=1, d=64, W=8, K=8,
                     T=3, V=512, levels=3, C=16, n_items=200, zipf=None,
                     logit_sigma=2.0, q_dtype=F32, kv_dtype=F32, out_dtype=F32),
    "qwen06b": Workload("qwen06b", R=1, prompt_lens=[2048], Hq=16, Hkv=8, d=128,
                        W=50, K=50, T=3, V=151936, levels=3, C=8192,
                        n_items=1_000_000, zipf=1.1, logit_sigma=2.0),
    "onerec17b": Workload("onerec17b", R=4, prompt_lens=[4096] * 4, Hq=16, Hkv=8,
                          d=128, W=512, K=512, T=3, V=151936, levels=3, C=8192,
                          n_items=4_000_000, zipf=1.1, logit_sigma=2.0),
    "fp8kv": Workload("fp8kv", R=4, prompt_lens=None, p_range=(512, 8192), Hq=16,
                      Hkv=8, d=128, W=1000, K=128, T=4, V=151936, levels=4,
                      C=4096, n_items=2_000_000, zipf=1.1, logit_sigma=3.0,
                      spike_p=0.01, spike_val=8.0, kv_dtype=E4M3),
    "openvocab": Workload("openvocab", R=2, prompt_lens=[1024] * 2, Hq=16, Hkv=8,
                          d=128, W=5000, K=5000, T=32, V=151936, levels=0, C=0,
                          n_items=0, zipf=None, logit_sigma=2.0),
}

# stream ids (one per tensor kind)
S_PLEN, S_CATALOG, S_Q, S_SK, S_SV, S_UK, S_UV, S_LOGIT, S_SPIKE, S_STATE = range(10)


def _np_rng(seed: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=[(seed << 32) | stream, sub]))


def _torch_gen(seed: int, stream: int, sub: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    s = (seed * 1_000_003 + stream) * 65_537 + sub
    if torch.device(device).type == "cpu":
        # the CPU generator keeps only the low 32 bits of its seed, and `sub`
        # carries the decode step above bit 31: fold the high half in
        s = ((s & 0xFFFFFFFF) ^ (((s >> 32) * 0x9E3779B1) & 0xFFFFFFFF))
    g.manual_seed(s)
    return g


def prompt_lens(wl: Workload) -> np.ndarray:
    if wl.prompt_lens is not None:
        return np.asarray(wl.prompt_lens, dtype=np.int64)
    lo, hi = wl.p_range
    return _np_rng(wl.seed, S_PLEN).integers(lo, hi + 1, size=wl.R).astype(np.int64)


def prompt_offsets(wl: Workload) -> np.ndarray:
    p = prompt_lens(wl)
    return np.concatenate([[0], np.cumsum(p)]).astype(np.int32)


def catalog(wl: Workload) -> np.ndarray:
    """[n_items, levels] int32 codes: distinct tuples, first n_items in draw order.

    Codes per level are i.i.d.; Zipf(s) draws code c with P(c) ~ (c+1)^-s,
    otherwise codes are uniform on [0, C).
    """
    if wl.levels == 0:
        return np.zeros((0, 0), dtype=np.int32)
    rng = _np_rng(wl.seed, S_CATALOG)
    if wl.zipf is None:
        cdf = None
    else:
        w = (np.arange(wl.C, dtype=np.float64) + 1.0) ** (-wl.zipf)
        cdf = np.cumsum(w) / w.sum()
    keys = np.zeros(0, dtype=np.int64)
    first = np.zeros(0, dtype=np.int64)
    bits = int(np.ceil(np.log2(max(wl.C, 2))))
    drawn = 0
    while True:
        n_draw = max(2 * (wl.n_items - len(first)), 1024)
        if cdf is None:
            codes = rng.integers(0, wl.C, size=(n_draw, wl.levels))
        else:
            u = rng.random(size=(n_draw, wl.levels))
            codes = np.minimum(np.searchsorted(cdf, u, side="right"), wl.C - 1)
        k = np.zeros(n_draw, dtype=np.int64)
        for lv in range(wl.levels):
            k = (k << bits) | codes[:, lv].astype(np.int64)
        keys = np.concatenate([keys, k])
        drawn += n_draw
        _, idx = np.unique(keys, return_index=True)
        first = np.sort(idx)
        if len(first) >= wl.n_items:
            first = first[: wl.n_items]
            break
    sel = keys[first]
    out = np.zeros((wl.n_items, wl.levels), dtype=np.int32)
    for lv in reversed(range(wl.levels)):
        out[:, lv] = (sel & ((1 << bits) - 1)).astype(np.int32)
        sel = sel >> bits
    return out


def _randn(shape, seed, stream, sub, device, dtype=torch.float32):
    g = _torch_gen(seed, stream, sub, device)
    return torch.randn(shape, generator=g, device=device, dtype=dtype)


def kv_scales(wl: Workload, device="cpu"):
    """Per-kv-head fp8 scales (amax / 448 over the shared KV of all requests)."""
    sk, sv = _shared_kv_f32(wl, device)
    ks = sk.abs().amax(dim=(0, 2)) / E4M3_MAX
    vs = sv.abs().amax(dim=(0, 2)) / E4M3_MAX
    return ks.float(), vs.float()


def _shared_kv_f32(wl: Workload, device):
    total = int(prompt_offsets(wl)[-1])
    sk = _randn((total, wl.Hkv, wl.d), wl.seed, S_SK, 0, device)
    sv = _randn((total, wl.Hkv, wl.d), wl.seed, S_SV, 0, device)
    return sk, sv


def _quant(x: torch.Tensor, dtype: int, scale: torch.Tensor | None):
    if dtype == F32:
        return x.float()
    if dtype == BF16:
        return x.to(torch.bfloat16)
    # e4m3: divide by the per-head scale, saturate to the finite range, round-nearest-even
    y = x / scale.view(1, -1, 1)
    y = y.clamp(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn)


def attention_inputs(wl: Workload, step: int, device="cpu"):
    """Q for one decode step plus the (step-independent) KV pools.

    Returns dict with
      q          [R, W, Hq, d]       q_dtype (fp32 or bf16)
      shared_k/v [sum P, Hkv, d]     kv_dtype
      unshared_k/v [R, T*W, Hkv, d]  kv_dtype (the slot pool; slot t*W+j holds
                                     the K/V of the token picked at step t by beam j)
      k_scale/v_scale [Hkv] fp32 (ones unless e4m3)
      prompt_offsets [R+1] int32
    """
    q = _randn((wl.R, wl.W, wl.Hq, wl.d), wl.seed, S_Q, step, device)
    q = q.float() if wl.q_dtype == F32 else q.to(torch.bfloat16)
    sk, sv = _shared_kv_f32(wl, device)
    uk = _randn((wl.R, wl.T * wl.W, wl.Hkv, wl.d), wl.seed, S_UK, 0, device)
    uv = _randn((wl.R, wl.T * wl.W, wl.Hkv, wl.d), wl.seed, S_UV, 0, device)
    if wl.kv_dtype == E4M3:
        ks = sk.abs().amax(dim=(0, 2)) / E4M3_MAX
        vs = sv.abs().amax(dim=(0, 2)) / E4M3_MAX
    else:
        ks = torch.ones(wl.Hkv, device=device)
        vs = torch.ones(wl.Hkv, device=device)
    return dict(
        q=q,
        shared_k=_quant(sk, wl.kv_dtype, ks), shared_v=_quant(sv, wl.kv_dtype, vs),
        unshared_k=_quant(uk, wl.kv_dtype, ks), unshared_v=_quant(uv, wl.kv_dtype, vs),
        k_scale=ks.float().contiguous(), v_scale=vs.float().contiguous(),
        prompt_offsets=torch.from_numpy(prompt_offsets(wl)).to(device),
    )


def logits(wl: Workload, step: int, rows: int | None = None, device="cpu"):
    """fp32 logits [R, rows, V] for decode step ``step`` (rows defaults to W).

    N(0, sigma) plus, where the workload has them, Bernoulli(spike_p) * spike_val.
    Rows are drawn in blocks of 64 with one generator per block, so
    ``logit_rows`` can regenerate any few rows of a multi-GB step alone.
    """
    rows = wl.W if rows is None else rows
    return torch.stack([logit_rows(wl, step, r, 0, rows, device) for r in range(wl.R)])


def logit_rows(wl: Workload, step: int, r: int, b0: int, b1: int, device="cpu"):
    """Rows b0..b1-1 of request r's step-``step`` logits (same values as ``logits``)."""
    parts = []
    for blk in range(b0 // 64, (b1 + 63) // 64):
        x = _logit_block64(wl, step, r, blk, device)
        lo = max(b0, blk * 64) - blk * 64
        hi = min(b1, blk * 64 + 64) - blk * 64
        parts.append(x[lo:hi])
    if not parts:
        return torch.zeros((0, wl.V), device=device)
    return torch.cat(parts)


def _logit_block64(wl, step, r, blk, device):
    sub = ((step * 4096 + r) << 20) | blk
    x = _randn((64, wl.V), wl.seed, S_LOGIT, sub, device) * wl.logit_sigma
    if wl.spike_p > 0:
        g = _torch_gen(wl.seed, S_SPIKE, sub, device)
        u = torch.rand((64, wl.V), generator=g, device=device)
        x = x + (u < wl.spike_p).float() * wl.spike_val
    return x


def steady_state(wl: Workload, items: np.ndarray, level: int, seed_sub: int = 0):
    """A decode state with all W beams live, for timing one step in isolation.

    Each beam sits at the level-``level`` node of a random catalog item's
    prefix (returned as the prefix codes; the caller maps them to node ids),
    with a random cumulative score and a random ancestry in the slot pool.
    Returns dict(prefix [R, W, level] int32, cum [R, W] fp32,
                 slot [R, W, T] int32, n_live [R] int32).
    """
    rng = _np_rng(wl.seed, S_STATE, seed_sub)
    R, W, T = wl.R, wl.W, wl.T
    if wl.levels > 0:
        pick = rng.integers(0, items.shape[0], size=(R, W))
        prefix = items[pick][:, :, :level].astype(np.int32)
    else:
        prefix = np.zeros((R, W, 0), dtype=np.int32)
    cum = (-rng.random(size=(R, W)) * 4.0 * level).astype(np.float32)
    slot = np.full((R, W, T), -1, dtype=np.int32)
    for t in range(level):
        slot[:, :, t] = t * W + rng.integers(0, W, size=(R, W))
    n_live = np.full(R, W, dtype=np.int32)
    return dict(prefix=prefix, cum=cum, slot=slot, n_live=n_live)
