"""C ABI checks that need no GPU: the library loads, exports every entry
point the header declares, validates arguments on the host and sizes its
workspaces.  No call here launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beamdec.h")


@pytest.fixture(scope="module")
def L():
    from wide_beam_generative_gb300 import build as b
    b.build()
    from wide_beam_generative_gb300 import beamdec
    return beamdec.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(beam\w*)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"beam_select", "beam_attn_decode", "beam_trie_build"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_error_strings(L):
    from wide_beam_generative_gb300 import beamdec as bd
    assert bd.error_string(0) == "ok"
    for s in range(-7, 0):
        assert bd.error_string(s) != "unknown status"
    assert L.beamdec_version().decode().count(".") == 2


FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: validation fails first
# distinct fake outputs (an output equal to its input is rejected as aliasing)
CUM_OUT, NODE_OUT, NLIVE_OUT, SLOT_OUT = (ctypes.c_void_p(v) for v in (0x4000, 0x5000, 0x6000, 0x2000))


def _select(L, **kw):
    args = dict(logits=FAKE, row_stride=512, lse_in=None, cum=FAKE, node=FAKE, n_live=FAKE,
                slot_in=FAKE, trie=None, level=0, step=0, R=1, W=8, K=8, V=512, T=3,
                tokens=FAKE, parents=FAKE, cum_out=CUM_OUT, lse_out=None, node_out=NODE_OUT,
                n_live_out=NLIVE_OUT, slot_out=SLOT_OUT, ws=FAKE, ws_bytes=0, stream=None)
    args.update(kw)
    return L.beam_select(*args.values())


def test_select_validation(L):
    from wide_beam_generative_gb300 import beamdec as bd
    assert _select(L, logits=None) == bd.ERR_INVALID_ARG
    assert _select(L, W=0) == bd.ERR_INVALID_ARG
    assert _select(L, step=3) == bd.ERR_INVALID_ARG
    assert _select(L, row_stride=100) == bd.ERR_INVALID_ARG
    assert _select(L, step=1, slot_in=None) == bd.ERR_INVALID_ARG
    assert _select(L, slot_out=FAKE) == bd.ERR_INVALID_ARG          # aliasing slot_in
    assert _select(L, cum_out=FAKE) == bd.ERR_INVALID_ARG           # aliasing cum_in
    assert _select(L, n_live_out=FAKE) == bd.ERR_INVALID_ARG        # aliasing n_live_in
    assert _select(L, node_out=FAKE) == bd.ERR_INVALID_ARG          # aliasing node_in
    assert _select(L, W=9000) == bd.ERR_UNSUPPORTED
    assert _select(L, V=300000, row_stride=300000) == bd.ERR_UNSUPPORTED
    assert _select(L, ws=ctypes.c_void_p(0x1010)) == bd.ERR_INVALID_ARG   # not 256-aligned
    assert _select(L, ws_bytes=16) == bd.ERR_WORKSPACE


def test_select_workspace_size(L):
    from wide_beam_generative_gb300 import beamdec as bd
    small = bd.beam_select_workspace_size(1, 8, 8, 512)
    big = bd.beam_select_workspace_size(4, 512, 512, 151936)
    assert big >= 4 * 512 * 512 * 8 > small > 0
    with pytest.raises(bd.BeamdecError):
        bd.beam_select_workspace_size(1, 9000, 8, 512)


def _attn(L, **kw):
    args = dict(q=FAKE, sk=FAKE, sv=FAKE, off=FAKE, maxp=256, rows=256, uk=FAKE, uv=FAKE, slot=FAKE,
                n_live=FAKE, step=0, R=1, W=8, Hq=2, Hkv=1, d=64, T=3, qd=0, kvd=0, od=0,
                ks=None, vs=None, sm=0.0, out=FAKE, ws=FAKE, ws_bytes=0, stream=None)
    args.update(kw)
    return L.beam_attn_decode(*args.values())


def test_attention_validation(L):
    from wide_beam_generative_gb300 import beamdec as bd
    assert _attn(L, q=None) == bd.ERR_INVALID_ARG
    assert _attn(L, Hq=3, Hkv=2) == bd.ERR_INVALID_ARG
    assert _attn(L, d=96) == bd.ERR_UNSUPPORTED
    assert _attn(L, Hq=34, Hkv=2) == bd.ERR_UNSUPPORTED                # group of 17
    assert _attn(L, qd=1, kvd=0, od=1) == bd.ERR_UNSUPPORTED            # bf16 q with fp32 KV
    assert _attn(L, qd=7) == bd.ERR_INVALID_ARG
    assert _attn(L, qd=1, kvd=2, od=1) == bd.ERR_INVALID_ARG            # e4m3 without scales
    assert _attn(L, step=3) == bd.ERR_INVALID_ARG
    assert _attn(L, maxp=256, sk=None) == bd.ERR_INVALID_ARG
    assert _attn(L, rows=100) == bd.ERR_INVALID_ARG                     # fewer rows than a prompt
    assert _attn(L) == bd.ERR_WORKSPACE
    n = bd.beam_attn_workspace_size(4, 512, 16, 8, 128, 4096, bd.BF16)
    assert n >= 4 * 512 * 16 * 128 * 4


def test_trie_validation_before_any_device_call(L):
    from wide_beam_generative_gb300 import beamdec as bd
    import numpy as np
    with pytest.raises(bd.BeamdecError) as e:
        bd.beam_trie_build(np.array([[0, 1, 16]]), [16, 16, 16], [0, 16, 32], 512)
    assert e.value.status == bd.ERR_INVALID_ARG                          # code 16 >= C
    with pytest.raises(bd.BeamdecError) as e:
        bd.beam_trie_build(np.array([[0, 1, 2]]), [16, 16, 16], [0, 16, 500], 512)
    assert e.value.status == bd.ERR_INVALID_ARG                          # range past vocab
    with pytest.raises(bd.BeamdecError) as e:
        bd.beam_trie_build(np.zeros((1, 9), np.int32), [2] * 9, [0] * 9, 512)
    assert e.value.status == bd.ERR_UNSUPPORTED                          # > 8 levels


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from wide_beam_generative_gb300 import beamdec as bd
    monkeypatch.setattr(bd, "_lib", None)
    monkeypatch.setattr(bd, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        bd.lib()


def test_static_select_rejects_oversized_shapes_on_host(L):
    from wide_beam_generative_gb300 import beamdec as bd
    fake = ctypes.c_void_p(0x1000)
    rc = L.beam_select_static(fake, 151936, None, fake, fake, fake, fake, None, 0, 0,
                              2, 5000, 5000, 151936, 2, fake, fake, CUM_OUT, None, NODE_OUT, NLIVE_OUT,
                              SLOT_OUT, None)
    assert rc == bd.ERR_UNSUPPORTED


def test_gumbel_select_validates_temperature_on_host(L):
    from wide_beam_generative_gb300 import beamdec as bd
    args = [FAKE, 512, None, FAKE, FAKE, FAKE, FAKE, None, 0, 0, 1, 8, 8, 512, 3]
    outs = [FAKE, FAKE, CUM_OUT, None, NODE_OUT, NLIVE_OUT, SLOT_OUT, FAKE, 0, None]
    for t in (0.0, -1.0, float("nan"), float("inf"), 1e-40):
        assert L.beam_select_gumbel(*args, t, 7, *outs) == bd.ERR_INVALID_ARG, t
    # a valid temperature reaches the same shape checks as beam_select
    assert L.beam_select_gumbel(*args, 0.7, 7, *outs) == bd.ERR_WORKSPACE


def test_dense_trie_validation_before_any_device_call(L):
    from wide_beam_generative_gb300 import beamdec as bd
    assert L.beam_trie_make_dense(None, 0, None) == bd.ERR_INVALID_ARG
    assert L.beam_trie_drop_dense(None, 0) == bd.ERR_INVALID_ARG
    assert L.beam_trie_export_dense(None, 0, None, None) == bd.ERR_INVALID_ARG


def test_fixed_lse_select_validates_on_host(L):
    from wide_beam_generative_gb300 import beamdec as bd
    head = [FAKE, 512]
    rest = [FAKE, FAKE, FAKE, FAKE, None, 0, 0, 1, 8, 8, 512, 3]
    outs = [FAKE, FAKE, CUM_OUT, None, NODE_OUT, NLIVE_OUT, SLOT_OUT, FAKE, 0, None]
    # score_lse is required
    assert L.beam_select_fixed_lse(*head, None, *rest, 0.0, 0, *outs) == bd.ERR_INVALID_ARG
    # temperature 0 (deterministic) or a valid Gumbel temperature; nothing else
    for t in (-1.0, float("nan"), float("inf"), 1e-40):
        assert L.beam_select_fixed_lse(*head, FAKE, *rest, t, 0, *outs) == bd.ERR_INVALID_ARG, t
    for t in (0.0, 0.7):   # valid: reaches the same shape checks as beam_select
        assert L.beam_select_fixed_lse(*head, FAKE, *rest, t, 0, *outs) == bd.ERR_WORKSPACE


def _splits_from_workspace(bd, R, W, Hq, Hkv, d, P):
    """Prompt splits the attention planner chose, read back from the
    workspace size (bf16 KV: header + per split and query row an (m, l)
    pair and a d-float partial output, each array 256-byte padded)."""
    rows1 = R * Hkv * W * (Hq // Hkv)
    n = bd.beam_attn_workspace_size(R, W, Hq, Hkv, d, P, bd.BF16)
    pad = lambda x: (x + 255) // 256 * 256
    for s in range(1, 17):
        if 256 + 2 * pad(rows1 * 4 * s) + pad(rows1 * d * 4 * s) == n:
            return s
    raise AssertionError(f"workspace size {n} matches no split count")


def test_attention_planner_split_choices(L):
    """The split model's choices on the benchmarked shapes: one split (the
    merge fused in the shared stage) where the CTAs already fill the GPU,
    eight for 1 x 50 beams over 2048 keys (measured 46.0 us per step against
    50.0 at sixteen and 47.8 at four), and the CUDA-core stage's split of a
    d = 64 prompt."""
    from wide_beam_generative_gb300 import beamdec as bd
    assert _splits_from_workspace(bd, 4, 512, 16, 8, 128, 4096) == 1      # 4 x 512, prompts 4096
    assert _splits_from_workspace(bd, 2, 5000, 16, 8, 128, 1024) == 1     # 2 x 5000, prompts 1024
    assert _splits_from_workspace(bd, 1, 50, 16, 8, 128, 2048) == 8       # 1 x 50, prompt 2048
    assert _splits_from_workspace(bd, 1, 8, 2, 1, 64, 256) == 2           # d = 64, CUDA cores
    assert _splits_from_workspace(bd, 1, 50, 16, 8, 128, 128) == 1        # a single chunk


def _prep(L, **kw):
    args = dict(sk=FAKE, sv=FAKE, off=FAKE, maxp=256, rows=256, R=1, W=8, Hq=16, Hkv=8, d=128, kvd=2,
                ws=FAKE, ws_bytes=0, stream=None)
    args.update(kw)
    return L.beam_attn_prepare_prompt(*args.values())


def test_prepare_prompt_validation(L):
    """beam_attn_prepare_prompt refuses bad arguments on the host and has
    nothing to do for KV types without a bf16 copy (no launch either way);
    the prepared kv type shares the e4m3 workspace layout."""
    from wide_beam_generative_gb300 import beamdec as bd
    assert _prep(L, off=None) == bd.ERR_INVALID_ARG
    assert _prep(L, ws=None) == bd.ERR_INVALID_ARG
    assert _prep(L, kvd=3) == bd.ERR_INVALID_ARG                        # the prepared type is a decode type
    assert _prep(L, kvd=-1) == bd.ERR_INVALID_ARG
    assert _prep(L, d=96) == bd.ERR_UNSUPPORTED
    assert _prep(L, rows=100) == bd.ERR_INVALID_ARG                     # fewer rows than a prompt
    assert _prep(L, sk=None) == bd.ERR_INVALID_ARG
    assert _prep(L, ws=ctypes.c_void_p(0x1010)) == bd.ERR_INVALID_ARG   # workspace not 256-byte aligned
    assert _prep(L, kvd=1) == bd.OK                                     # bf16: nothing to prepare
    assert _prep(L) == bd.ERR_WORKSPACE
    for shape in ((4, 1000, 16, 8, 128, 5212), (1, 50, 16, 8, 128, 2048), (1, 8, 2, 1, 64, 256)):
        assert bd.beam_attn_workspace_size(*shape, bd.E4M3_PREPARED) == \
            bd.beam_attn_workspace_size(*shape, bd.E4M3)
    assert _attn(L, qd=1, kvd=3, od=1) == bd.ERR_INVALID_ARG            # prepared e4m3 without scales
    assert _attn(L, qd=1, kvd=4, od=1) == bd.ERR_INVALID_ARG


def _lmh(L, **kw):
    args = dict(hidden=FAKE, weight=FAKE, rows=2048, hidden_dim=2048, V=151936, w0=8192, wlen=8192,
                lse=FAKE, logits=FAKE, stride=8192 * 2, ws=FAKE, ws_bytes=0, stream=None)
    args.update(kw)
    return L.beam_lmhead_lse(*args.values())


def test_lmhead_validation_on_host(L):
    """beam_lmhead_lse checks its pointers, shapes, window, alignment and
    workspace size before any device call (every case here fails one of
    those checks, so nothing is launched); its workspace size grows with
    the rows and the vocabulary."""
    from wide_beam_generative_gb300 import beamdec as bd
    for k in ("hidden", "weight", "lse", "ws"):
        assert _lmh(L, **{k: None}) == bd.ERR_INVALID_ARG, k
    assert _lmh(L, rows=0) == bd.ERR_INVALID_ARG
    assert _lmh(L, V=0) == bd.ERR_INVALID_ARG
    assert _lmh(L, hidden_dim=32) == bd.ERR_INVALID_ARG                     # below one 64-wide slice
    assert _lmh(L, w0=-1) == bd.ERR_INVALID_ARG
    assert _lmh(L, wlen=-1) == bd.ERR_INVALID_ARG
    assert _lmh(L, w0=151936 - 100, wlen=101) == bd.ERR_INVALID_ARG          # window past the vocabulary
    assert _lmh(L, hidden_dim=2048 + 32) == bd.ERR_UNSUPPORTED               # not a multiple of 64
    assert _lmh(L, V=(1 << 18) + 1) == bd.ERR_UNSUPPORTED                    # above the largest vocabulary
    assert _lmh(L, logits=None) == bd.ERR_INVALID_ARG                        # a window needs its buffer
    assert _lmh(L, stride=8192 + 8191) == bd.ERR_INVALID_ARG                 # row shorter than the window's end
    assert _lmh(L, hidden=ctypes.c_void_p(0x1008)) == bd.ERR_INVALID_ARG     # not 16-byte aligned
    assert _lmh(L, weight=ctypes.c_void_p(0x1008)) == bd.ERR_INVALID_ARG
    assert _lmh(L, ws=ctypes.c_void_p(0x1010)) == bd.ERR_INVALID_ARG         # not 256-byte aligned
    assert _lmh(L) == bd.ERR_WORKSPACE                                       # zero workspace bytes
    assert _lmh(L, wlen=0, logits=None) == bd.ERR_WORKSPACE                  # lse only: no window buffer needed
    size = ctypes.c_size_t()
    assert L.beam_lmhead_workspace_size(0, 151936, ctypes.byref(size)) == bd.ERR_INVALID_ARG
    assert L.beam_lmhead_workspace_size(2048, 0, ctypes.byref(size)) == bd.ERR_INVALID_ARG
    assert L.beam_lmhead_workspace_size(2048, 151936, None) == bd.ERR_INVALID_ARG
    sizes = []
    for rows, V in ((128, 512), (2048, 512), (2048, 151936)):
        assert L.beam_lmhead_workspace_size(rows, V, ctypes.byref(size)) == bd.OK
        sizes.append(size.value)
    assert 0 < sizes[0] <= sizes[1] <= sizes[2]


def test_profile_and_status_calls_on_host(L):
    """The profiling, status and trie-info entry points refuse bad arguments
    without touching a device; kernel ids name the kernels in the order the
    header documents; with nothing recorded a read returns zero launches
    (no event is created while recording is off)."""
    from wide_beam_generative_gb300 import beamdec as bd
    names = ["bd_expand_kernel", "bd_global_kernel", "bd_attn_shared_simt_kernel",
             "bd_attn_shared_tc_kernel", "bd_attn_merge_kernel", "bd_kv_e4m3_to_bf16_kernel",
             "bd_stream_select_kernel", "bd_lmhead_kernel", "bd_lmhead_lse_kernel", "bd_seed_kernel"]
    assert [L.beamdec_kernel_name(i).decode() for i in range(len(names))] == names
    assert L.beamdec_kernel_name(-1) == b"" and L.beamdec_kernel_name(len(names)) == b""
    assert L.beamdec_profile_enable(0) == bd.OK                   # off: creates nothing
    ms, n = ctypes.c_float(-1.0), ctypes.c_int(-1)
    for kid in range(len(names)):
        assert L.beamdec_profile_read(kid, ctypes.byref(ms), ctypes.byref(n)) == bd.OK
        assert (ms.value, n.value) == (0.0, 0)
    assert L.beamdec_profile_read(-1, ctypes.byref(ms), ctypes.byref(n)) == bd.ERR_INVALID_ARG
    assert L.beamdec_profile_read(len(names), ctypes.byref(ms), ctypes.byref(n)) == bd.ERR_INVALID_ARG
    assert L.beamdec_profile_read(0, None, ctypes.byref(n)) == bd.ERR_INVALID_ARG
    assert L.beamdec_profile_read(0, ctypes.byref(ms), None) == bd.ERR_INVALID_ARG
    st = ctypes.c_int32(7)
    assert L.beamdec_read_status(None, None, ctypes.byref(st)) == bd.ERR_INVALID_ARG
    assert L.beamdec_read_status(FAKE, None, None) == bd.ERR_INVALID_ARG
    assert st.value == 7                                          # untouched on refusal
    lv = ctypes.c_int(-1)
    assert L.beam_trie_info(None, ctypes.byref(lv), None, None, None, None, None) == bd.ERR_INVALID_ARG
    assert lv.value == -1
    L.beam_trie_free(None)                                        # a null handle is a no-op
