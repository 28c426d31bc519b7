"""Python binding of libbeamdec: argument marshalling only.

Every function here forwards torch tensors' device pointers and the current
CUDA stream to the C ABI declared in ``include/beamdec.h``; all computation
happens in the library's CUDA kernels.  There is no CPU or eager fallback: if
the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbeamdec.so")

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK, ERR_ALLOC = \
    -1, -2, -3, -4, -5, -6, -7
F32, BF16, E4M3 = 0, 1, 2
E4M3_PREPARED = 3   # kv dtype of a decode call whose prompt K/V the workspace holds as bf16
_DT = {torch.float32: F32, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3}

_lib = None

c_int, c_i64, c_sz, c_f, c_p = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_void_p
c_i32p = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "beamdec_error_string": (ctypes.c_char_p, [c_int]),
    "beamdec_version": (ctypes.c_char_p, []),
    "beamdec_read_status": (c_int, [c_p, c_p, c_i32p]),
    "beamdec_profile_enable": (c_int, [c_int]),
    "beamdec_profile_enable_mask": (c_int, [ctypes.c_uint]),
    "beamdec_profile_read": (c_int, [c_int, ctypes.POINTER(c_f), ctypes.POINTER(c_int)]),
    "beamdec_kernel_name": (ctypes.c_char_p, [c_int]),
    "beam_trie_build": (c_int, [c_p, c_i64, c_int, c_p, c_p, ctypes.c_int32, c_p, ctypes.POINTER(c_p)]),
    "beam_trie_free": (None, [c_p]),
    "beam_trie_info": (c_int, [c_p, ctypes.POINTER(c_int), c_i32p, ctypes.POINTER(c_i64),
                               c_p, c_p, c_p]),
    "beam_trie_export": (c_int, [c_p, c_int, ctypes.POINTER(c_p), ctypes.POINTER(c_p)]),
    "beam_select_workspace_size": (c_int, [c_int, c_int, c_int, c_int, ctypes.POINTER(c_sz)]),
    "beam_select": (c_int, [c_p, c_i64, c_p, c_p, c_p, c_p, c_p, c_p, c_int, c_int,
                            c_int, c_int, c_int, c_int, c_int,
                            c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "beam_select_gumbel": (c_int, [c_p, c_i64, c_p, c_p, c_p, c_p, c_p, c_p, c_int, c_int,
                                   c_int, c_int, c_int, c_int, c_int, c_f, ctypes.c_uint64,
                                   c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "beam_select_fixed_lse": (c_int, [c_p, c_i64, c_p, c_p, c_p, c_p, c_p, c_p, c_int, c_int,
                                      c_int, c_int, c_int, c_int, c_int, c_f, ctypes.c_uint64,
                                      c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]),
    "beam_trie_make_dense": (c_int, [c_p, c_int, c_p]),
    "beam_trie_drop_dense": (c_int, [c_p, c_int]),
    "beam_trie_export_dense": (c_int, [c_p, c_int, ctypes.POINTER(c_p), ctypes.POINTER(ctypes.c_int32)]),
    "beam_lmhead_workspace_size": (c_int, [c_int, c_int, ctypes.POINTER(c_sz)]),
    "beam_lmhead_lse": (c_int, [c_p, c_p, c_int, c_int, c_int, c_int, c_int, c_p, c_p, c_i64, c_p, c_sz,
                                c_p]),
    "beam_select_static": (c_int, [c_p, c_i64, c_p, c_p, c_p, c_p, c_p, c_p, c_int, c_int,
                                   c_int, c_int, c_int, c_int, c_int,
                                   c_p, c_p, c_p, c_p, c_p, c_p, c_p, c_p]),
    "beam_attn_workspace_size": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                         ctypes.POINTER(c_sz)]),
    "beam_attn_decode": (c_int, [c_p, c_p, c_p, c_p, c_int, c_i64, c_p, c_p, c_p, c_p, c_int,
                                 c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                 c_p, c_p, c_f, c_p, c_p, c_sz, c_p]),
    "beam_attn_prepare_prompt": (c_int, [c_p, c_p, c_p, c_int, c_i64, c_int, c_int, c_int, c_int, c_int,
                                         c_int, c_p, c_sz, c_p]),
}


class BeamdecError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {error_string(status)} ({status})")


def lib():
    """Loads libbeamdec.so (built in-tree by ``build.py``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbeamdec.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def error_string(status):
    return lib().beamdec_error_string(int(status)).decode()


def _check(status, where):
    if status != OK:
        raise BeamdecError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


class _DevArray:
    """Zero-copy view of a device int32 array owned by the library."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (int(n),), "typestr": "<i4",
                                         "data": (int(ptr), False), "version": 3}


class Trie:
    """Handle of a catalog trie in device memory (freed with the object)."""

    def __init__(self, handle):
        self._h = handle

    @property
    def handle(self):
        return self._h

    def info(self):
        L = lib()
        levels, vocab, n = c_int(), ctypes.c_int32(), c_i64()
        nodes = (c_i64 * 8)()
        edges = (c_i64 * 8)()
        mc = (ctypes.c_int32 * 8)()
        _check(L.beam_trie_info(self._h, ctypes.byref(levels), ctypes.byref(vocab), ctypes.byref(n),
                                nodes, edges, mc), "beam_trie_info")
        k = levels.value
        return dict(levels=k, vocab=vocab.value, n_items=n.value, n_nodes=list(nodes[:k]),
                    n_edges=list(edges[:k]), max_children=list(mc[:k]))

    def export(self, level):
        """(off, code) of one level as torch int32 CUDA tensors (copies)."""
        info = self.info()
        off, code = c_p(), c_p()
        _check(lib().beam_trie_export(self._h, level, ctypes.byref(off), ctypes.byref(code)),
               "beam_trie_export")
        o = torch.as_tensor(_DevArray(off.value, info["n_nodes"][level] + 1), device="cuda").clone()
        c = torch.as_tensor(_DevArray(code.value, info["n_edges"][level]), device="cuda").clone()
        return o, c

    def make_dense(self, level, stream=None):
        """Build dense child masks for `level`; selections then enumerate
        that level's candidates from them (without ``lse_in`` in two
        launches instead of one; results are identical)."""
        _check(lib().beam_trie_make_dense(self.handle, level, _stream(stream)), "beam_trie_make_dense")

    def drop_dense(self, level):
        _check(lib().beam_trie_drop_dense(self.handle, level), "beam_trie_drop_dense")

    def export_dense(self, level):
        """[n_nodes, words] int32 copy of the level's masks (bit c = code c), or None."""
        ptr, words = c_p(), ctypes.c_int32()
        _check(lib().beam_trie_export_dense(self.handle, level, ctypes.byref(ptr), ctypes.byref(words)),
               "beam_trie_export_dense")
        if not ptr.value:
            return None
        n_nodes = int(self.info()["n_nodes"][level])
        out = torch.empty((n_nodes, words.value), dtype=torch.int32, device="cuda")
        src = torch.as_tensor(_DevArray(ptr.value, n_nodes * words.value), device="cuda")
        out.copy_(src.view(n_nodes, words.value))
        return out

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.beam_trie_free(self._h)
            self._h = None


def beam_trie_build(items, codes_per_level, token_base, vocab, stream=None) -> Trie:
    """Canonical CSR trie of ``items`` [n, levels] (host int32 codes)."""
    items = np.ascontiguousarray(np.asarray(items, dtype=np.int32))
    cpl = np.ascontiguousarray(np.asarray(codes_per_level, dtype=np.int32))
    tb = np.ascontiguousarray(np.asarray(token_base, dtype=np.int32))
    h = c_p()
    st = _stream(stream) if torch.cuda.is_available() else c_p(0)
    _check(lib().beam_trie_build(items.ctypes.data, items.shape[0], items.shape[1], cpl.ctypes.data,
                                 tb.ctypes.data, int(vocab), st, ctypes.byref(h)), "beam_trie_build")
    return Trie(h)


def workspace(nbytes, device="cuda"):
    """Zero-filled, 256-byte aligned device workspace of ``nbytes``."""
    ws = torch.zeros(int(nbytes) + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + int(nbytes)]


def beam_select_workspace_size(R, W, K, V):
    n = c_sz()
    _check(lib().beam_select_workspace_size(R, W, K, V, ctypes.byref(n)), "beam_select_workspace_size")
    return n.value


def beam_attn_workspace_size(R, W, Hq, Hkv, d, max_prompt_len, kv_dtype):
    n = c_sz()
    _check(lib().beam_attn_workspace_size(R, W, Hq, Hkv, d, max_prompt_len, kv_dtype, ctypes.byref(n)),
           "beam_attn_workspace_size")
    return n.value


KERNELS = ["bd_expand_kernel", "bd_global_kernel", "bd_attn_shared_simt_kernel",
           "bd_attn_shared_tc_kernel", "bd_attn_merge_kernel", "bd_kv_e4m3_to_bf16_kernel",
           "bd_stream_select_kernel", "bd_lmhead_kernel", "bd_lmhead_lse_kernel", "bd_seed_kernel"]


def profile_enable(on=True, kernels=None):
    """Start (or stop) per-kernel event timing; `kernels` (names) limits it
    to those kernels."""
    if kernels is None:
        _check(lib().beamdec_profile_enable(1 if on else 0), "beamdec_profile_enable")
        return
    mask = 0
    for name in kernels:
        mask |= 1 << KERNELS.index(name)
    _check(lib().beamdec_profile_enable_mask(mask if on else 0), "beamdec_profile_enable_mask")


def profile_read():
    """{kernel name: (total ms, launches)} of the launches recorded since enable."""
    res = {}
    for k, name in enumerate(KERNELS):
        ms, n = c_f(), c_int()
        _check(lib().beamdec_profile_read(k, ctypes.byref(ms), ctypes.byref(n)), "beamdec_profile_read")
        res[name] = (ms.value, n.value)
    return res


def read_status(ws, stream=None):
    v = ctypes.c_int32()
    _check(lib().beamdec_read_status(_ptr(ws), _stream(stream), ctypes.byref(v)), "beamdec_read_status")
    return v.value


def beam_select(logits, cum, node, n_live, slot_in, trie, level, step, K, T=None,
                lse_in=None, out=None, ws=None, stream=None, want_lse=True, temperature=0.0, seed=0,
                score_lse=None):
    """One expansion step.  logits [R, W, V] fp32 (row b of request r at
    logits[r, b]); cum [R, W] fp32; node [R, W] int32 (ignored without trie);
    n_live [R] int32; slot_in [R, W, T] int32.  Returns a dict of output
    tensors: tokens, parents, cum_out, lse_out, node_out, n_live_out, slot_out.
    temperature > 0 selects by Gumbel top-k (beam_select_gumbel) with the
    64-bit ``seed``.  score_lse [R, W] fp32 runs the one-launch kernel with
    the candidates scored against these normalisers
    (beam_select_fixed_lse); lse_out still holds the kernel's own."""
    R, W = cum.shape
    V = logits.shape[-1]
    if logits.dim() != 3 or logits.shape[0] != R or logits.shape[1] != W or logits.stride(2) != 1 \
            or logits.stride(0) != W * logits.stride(1):
        raise ValueError("logits must be [R, W, V] with unit stride in V and rows packed per request")
    T = slot_in.shape[2] if T is None else T
    _need_cuda(cum, node, n_live, slot_in, lse_in, score_lse)
    if lse_in is not None and score_lse is not None:
        raise ValueError("lse_in and score_lse are exclusive")
    dev = cum.device
    if out is None:
        out = dict(tokens=torch.empty((R, W), dtype=torch.int32, device=dev),
                   parents=torch.empty((R, W), dtype=torch.int32, device=dev),
                   cum_out=torch.empty((R, W), dtype=torch.float32, device=dev),
                   lse_out=torch.empty((R, W), dtype=torch.float32, device=dev) if want_lse else None,
                   node_out=torch.empty((R, W), dtype=torch.int32, device=dev),
                   n_live_out=torch.empty((R,), dtype=torch.int32, device=dev),
                   slot_out=torch.empty((R, W, T), dtype=torch.int32, device=dev))
    if ws is None:
        ws = workspace(beam_select_workspace_size(R, W, K, V), dev)
    head = (_ptr(logits), logits.stride(1), _ptr(lse_in if score_lse is None else score_lse), _ptr(cum),
            _ptr(node), _ptr(n_live), _ptr(slot_in), trie.handle if trie is not None else None, level, step,
            R, W, K, V, T)
    tail = (_ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["cum_out"]), _ptr(out.get("lse_out")),
            _ptr(out["node_out"]), _ptr(out["n_live_out"]), _ptr(out["slot_out"]), _ptr(ws), ws.numel(),
            _stream(stream))
    if score_lse is not None:
        rc = lib().beam_select_fixed_lse(*head, float(temperature), int(seed) & (2 ** 64 - 1), *tail)
        _check(rc, "beam_select_fixed_lse")
    elif temperature > 0:
        rc = lib().beam_select_gumbel(*head, float(temperature), int(seed) & (2 ** 64 - 1), *tail)
        _check(rc, "beam_select_gumbel")
    else:
        rc = lib().beam_select(*head, *tail)
        _check(rc, "beam_select")
    return out


def beam_select_static(logits, cum, node, n_live, slot_in, trie, level, step, K, T=None,
                       lse_in=None, out=None, stream=None, want_lse=True):
    """beam_select with the library's fixed static scratch instead of a
    workspace (for callers that cannot allocate); same arguments and outputs."""
    R, W = cum.shape
    V = logits.shape[-1]
    if logits.dim() != 3 or logits.shape[0] != R or logits.shape[1] != W or logits.stride(2) != 1 \
            or logits.stride(0) != W * logits.stride(1):
        raise ValueError("logits must be [R, W, V] with unit stride in V and rows packed per request")
    T = slot_in.shape[2] if T is None else T
    _need_cuda(cum, node, n_live, slot_in, lse_in)
    dev = cum.device
    if out is None:
        out = dict(tokens=torch.empty((R, W), dtype=torch.int32, device=dev),
                   parents=torch.empty((R, W), dtype=torch.int32, device=dev),
                   cum_out=torch.empty((R, W), dtype=torch.float32, device=dev),
                   lse_out=torch.empty((R, W), dtype=torch.float32, device=dev) if want_lse else None,
                   node_out=torch.empty((R, W), dtype=torch.int32, device=dev),
                   n_live_out=torch.empty((R,), dtype=torch.int32, device=dev),
                   slot_out=torch.empty((R, W, T), dtype=torch.int32, device=dev))
    rc = lib().beam_select_static(_ptr(logits), logits.stride(1), _ptr(lse_in), _ptr(cum), _ptr(node),
                                  _ptr(n_live), _ptr(slot_in), trie.handle if trie is not None else None,
                                  level, step, R, W, K, V, T,
                                  _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["cum_out"]),
                                  _ptr(out.get("lse_out")), _ptr(out["node_out"]), _ptr(out["n_live_out"]),
                                  _ptr(out["slot_out"]), _stream(stream))
    _check(rc, "beam_select_static")
    return out


def beam_attn_prepare_prompt(shared_k, shared_v, prompt_offsets, max_prompt_len, W, Hq, ws, stream=None):
    """Writes the bf16 copy of e4m3 prompt K/V into the attention workspace
    ``ws`` (sized for these shapes), for later ``beam_attn_decode(...,
    prepared=True)`` calls on the same prompt; other KV types: nothing to do."""
    R = prompt_offsets.shape[0] - 1
    Hkv, d = shared_k.shape[1], shared_k.shape[2]
    _need_cuda(shared_k, shared_v, prompt_offsets, ws)
    rc = lib().beam_attn_prepare_prompt(_ptr(shared_k), _ptr(shared_v), _ptr(prompt_offsets),
                                        int(max_prompt_len), int(shared_k.shape[0]), R, int(W), int(Hq),
                                        Hkv, d, _DT[shared_k.dtype], _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "beam_attn_prepare_prompt")


def beam_attn_decode(q, shared_k, shared_v, prompt_offsets, max_prompt_len, unshared_k, unshared_v,
                     slot_table, n_live, step, k_scale=None, v_scale=None, sm_scale=0.0,
                     out=None, ws=None, stream=None, prepared=False):
    """Split-KV beam attention for one decode step; returns ``out``
    [R, W, Hq, d] (fp32 for fp32 q, else bf16).  ``prepared``: e4m3 KV whose
    prompt part ``beam_attn_prepare_prompt`` already copied into ``ws``."""
    R, W, Hq, d = q.shape
    Hkv = unshared_k.shape[2]
    T = slot_table.shape[2]
    _need_cuda(q, shared_k, shared_v, prompt_offsets, unshared_k, unshared_v, slot_table, n_live,
               k_scale, v_scale)
    qd, kvd = _DT[q.dtype], _DT[unshared_k.dtype]
    od = F32 if qd == F32 else BF16
    if prepared and kvd == E4M3:
        if ws is None:
            raise ValueError("prepared=True needs the workspace beam_attn_prepare_prompt wrote")
        kvd = E4M3_PREPARED
    if out is None:
        out = torch.empty((R, W, Hq, d), dtype=torch.float32 if od == F32 else torch.bfloat16,
                          device=q.device)
    if ws is None:
        ws = workspace(beam_attn_workspace_size(R, W, Hq, Hkv, d, max_prompt_len, kvd), q.device)
    shared_rows = shared_k.shape[0] if shared_k is not None else 0
    rc = lib().beam_attn_decode(_ptr(q), _ptr(shared_k), _ptr(shared_v), _ptr(prompt_offsets),
                                int(max_prompt_len), int(shared_rows), _ptr(unshared_k), _ptr(unshared_v),
                                _ptr(slot_table), _ptr(n_live), step, R, W, Hq, Hkv, d, T,
                                qd, kvd, od, _ptr(k_scale), _ptr(v_scale), float(sm_scale),
                                _ptr(out), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "beam_attn_decode")
    return out


class DecodeChain:
    """T decode steps (selection, then attention, per step) captured once as a
    single CUDA graph and replayed with no host work between steps.

    logits[t] [R, W, V] fp32 and q[t] [R, W, Hq, d] are the per-step inputs,
    resident on the device; the prompt KV and the slot pool of unshared KV
    are shared by all steps.  Every replay starts from one live beam per
    request (cum 0, trie root, empty slot rows), exactly as the eager chain
    does, and leaves step t's outputs in ``sel[t]`` (the beam_select dict)
    and ``out[t]`` (the attention output).  ``score_lse`` (optional, one
    [R, W] fp32 tensor per step) scores every step's candidates against
    those normalisers (beam_select_fixed_lse), for comparisons with a
    reference that rounds its own.  The C ABI makes this possible:
    its compute calls neither allocate nor synchronise the host, so graph
    capture records the same launches an eager call would make.
    """

    def __init__(self, logits, q, shared_k, shared_v, prompt_offsets, max_prompt_len,
                 unshared_k, unshared_v, trie, K, k_scale=None, v_scale=None, sm_scale=0.0,
                 score_lse=None):
        T = len(logits)
        R, W, V = logits[0].shape
        Hq, d = q[0].shape[2], q[0].shape[3]
        Hkv = unshared_k.shape[2]
        dev = logits[0].device
        self.T = T
        self._state0 = dict(cum=torch.zeros((R, W), dtype=torch.float32, device=dev),
                            node=torch.zeros((R, W), dtype=torch.int32, device=dev),
                            n_live=torch.ones((R,), dtype=torch.int32, device=dev),
                            slot=torch.full((R, W, T), -1, dtype=torch.int32, device=dev))
        self._state = {k: torch.empty_like(v) for k, v in self._state0.items()}
        self.sel = [dict(tokens=torch.empty((R, W), dtype=torch.int32, device=dev),
                         parents=torch.empty((R, W), dtype=torch.int32, device=dev),
                         cum_out=torch.empty((R, W), dtype=torch.float32, device=dev),
                         lse_out=torch.empty((R, W), dtype=torch.float32, device=dev),
                         node_out=torch.empty((R, W), dtype=torch.int32, device=dev),
                         n_live_out=torch.empty((R,), dtype=torch.int32, device=dev),
                         slot_out=torch.empty((R, W, T), dtype=torch.int32, device=dev))
                    for _ in range(T)]
        out_dt = torch.float32 if q[0].dtype == torch.float32 else torch.bfloat16
        self.out = [torch.empty((R, W, Hq, d), dtype=out_dt, device=dev) for _ in range(T)]
        self._ws_sel = workspace(beam_select_workspace_size(R, W, K, V), dev)
        self._ws_att = workspace(beam_attn_workspace_size(R, W, Hq, Hkv, d, max_prompt_len,
                                                          _DT[unshared_k.dtype]), dev)
        # the prompt K/V is fixed for the chain: e4m3 is dequantised once here
        # and every step reads the copy (other KV types: nothing to do)
        beam_attn_prepare_prompt(shared_k, shared_v, prompt_offsets, max_prompt_len, W, Hq, self._ws_att)

        def chain():
            for k, v in self._state0.items():
                self._state[k].copy_(v)
            st = self._state
            for t in range(T):
                o = beam_select(logits[t], st["cum"], st["node"], st["n_live"], st["slot"], trie, t, t, K,
                                out=self.sel[t], ws=self._ws_sel,
                                score_lse=None if score_lse is None else score_lse[t])
                beam_attn_decode(q[t], shared_k, shared_v, prompt_offsets, max_prompt_len, unshared_k,
                                 unshared_v, o["slot_out"], o["n_live_out"], t, k_scale=k_scale,
                                 v_scale=v_scale, sm_scale=sm_scale, out=self.out[t], ws=self._ws_att,
                                 prepared=True)
                st = dict(cum=o["cum_out"], node=o["node_out"], n_live=o["n_live_out"], slot=o["slot_out"])

        # one eager pass on a side stream (first-use setup such as kernel
        # attributes happens outside the capture), then the capture itself
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            chain()
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            chain()

    def replay(self):
        """Run the T steps on the current stream (asynchronously)."""
        self.graph.replay()

    def status(self):
        """Device-side status words of the selection and attention workspaces."""
        return read_status(self._ws_sel), read_status(self._ws_att)


def beam_lmhead_workspace_size(rows, V):
    n = c_sz()
    _check(lib().beam_lmhead_workspace_size(rows, V, ctypes.byref(n)), "beam_lmhead_workspace_size")
    return n.value


def beam_lmhead_lse(hidden, weight, window_start=0, window_len=0, lse_out=None, logits_out=None, ws=None,
                    stream=None):
    """LM head with the log-sum-exp fused in: hidden [rows, H] bf16, weight
    [V, H] bf16.  Returns (lse [rows] fp32, logits [rows, V] fp32 of which
    only the window's columns are written, or None without a window)."""
    _need_cuda(hidden, weight)
    rows, H = hidden.shape
    V = weight.shape[0]
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16 or weight.shape[1] != H:
        raise ValueError("hidden [rows, H] and weight [V, H] must be bf16")
    dev = hidden.device
    if lse_out is None:
        lse_out = torch.empty(rows, dtype=torch.float32, device=dev)
    if window_len and logits_out is None:
        logits_out = torch.empty((rows, V), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(beam_lmhead_workspace_size(rows, V), dev)
    stride = logits_out.stride(0) if logits_out is not None else 0
    rc = lib().beam_lmhead_lse(_ptr(hidden), _ptr(weight), rows, H, V, window_start, window_len, _ptr(lse_out),
                               _ptr(logits_out), stride, _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "beam_lmhead_lse")
    return lse_out, logits_out
