"""Beam attention for one decode step (oracle side).

"Generative recommendation design" §4.2.1 splits the KV cache into shared KV
(the prompt's prefill KV, stored once and used by every beam of the request)
and unshared KV (one entry per decode token per beam); §4.2.2 computes the
attention in three stages (shared, unshared, online-softmax merge) only to
reach the same result as attention over the concatenated sequence faster.
The oracle therefore computes the plain definition:

for request r, live beam j < n_live[r], query head h (kv head g = h // G):
    keys/values = prompt rows 0..P_r-1 of head g, followed by the unshared
                  slots slot[r, j, 0..step] of head g (the beam's ancestry,
                  oldest first), all decoded exactly to float64;
    o[r, j, h]  = sum_i softmax_i(scale * q . k_i) v_i       (float64)
with ``scale`` = 1/sqrt(d) unless given.  Rows j >= n_live[r] are zero.

``attention_split`` restates the three-stage form (shared chunks, unshared,
merge) for the test that pins the two against each other.
"""
import numpy as np

from .dequant import to_f64


def _decode_inputs(inp):
    """float64 views of q and the KV pools (inp: dict of numpy arrays / raw bits)."""
    kvd = int(inp["kv_dtype"])
    qd = int(inp["q_dtype"])
    q = to_f64(inp["q"], qd)
    ks, vs = inp.get("k_scale"), inp.get("v_scale")
    sk = to_f64(inp["shared_k"], kvd, ks)
    sv = to_f64(inp["shared_v"], kvd, vs)
    uk = to_f64(inp["unshared_k"], kvd, ks)
    uv = to_f64(inp["unshared_v"], kvd, vs)
    return q, sk, sv, uk, uv


def _softmax_rows(s):
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def attention_decode(inp, slot, n_live, step, scale=None, beams=None):
    """Float64 attention output [R, W, Hq, d] over prompt + ancestor KV.

    ``inp`` holds q [R,W,Hq,d], shared_k/v [sumP,Hkv,d], unshared_k/v
    [R,T*W,Hkv,d] (raw storage: float32, or uint16 bf16 bits, or uint8 e4m3
    bits), k_scale/v_scale [Hkv], prompt_offsets [R+1], q_dtype, kv_dtype.
    ``beams``: optional list of (r, j) to compute (others stay zero).
    """
    q, sk, sv, uk, uv = _decode_inputs(inp)
    R, W, Hq, d = q.shape
    Hkv = sk.shape[1]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    off = np.asarray(inp["prompt_offsets"], dtype=np.int64)
    out = np.zeros((R, W, Hq, d))
    todo = beams if beams is not None else [(r, j) for r in range(R) for j in range(int(n_live[r]))]
    for r, j in todo:
        if j >= int(n_live[r]):
            continue
        slots = np.asarray(slot[r, j, : step + 1], dtype=np.int64)
        for g in range(Hkv):
            keys = np.concatenate([sk[off[r]:off[r + 1], g, :], uk[r, slots, g, :]], axis=0)
            vals = np.concatenate([sv[off[r]:off[r + 1], g, :], uv[r, slots, g, :]], axis=0)
            qh = q[r, j, g * G:(g + 1) * G, :]            # [G, d]
            p = _softmax_rows(scale * (qh @ keys.T))     # [G, P + L]
            out[r, j, g * G:(g + 1) * G, :] = p @ vals
    return out


def attention_split(inp, slot, n_live, step, chunk=64, scale=None):
    """Three-stage restatement: per prompt chunk and for the unshared tail, the
    partial triple (m, l, o) with o normalised by l; then the online-softmax
    merge m* = max m_i, l* = sum l_i e^(m_i - m*), o* = sum o_i l_i e^(m_i - m*) / l*.
    Used only to pin ``attention_decode`` (the two must agree to rounding)."""
    q, sk, sv, uk, uv = _decode_inputs(inp)
    R, W, Hq, d = q.shape
    Hkv = sk.shape[1]
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    off = np.asarray(inp["prompt_offsets"], dtype=np.int64)
    out = np.zeros((R, W, Hq, d))

    def partial(qh, keys, vals):
        s = scale * (qh @ keys.T)
        m = s.max(axis=-1)
        e = np.exp(s - m[:, None])
        l = e.sum(axis=-1)
        return m, l, (e @ vals) / l[:, None]

    for r in range(R):
        for j in range(int(n_live[r])):
            slots = np.asarray(slot[r, j, : step + 1], dtype=np.int64)
            for g in range(Hkv):
                qh = q[r, j, g * G:(g + 1) * G, :]
                parts = []
                for c0 in range(off[r], off[r + 1], chunk):
                    c1 = min(off[r + 1], c0 + chunk)
                    parts.append(partial(qh, sk[c0:c1, g], sv[c0:c1, g]))
                parts.append(partial(qh, uk[r, slots, g], uv[r, slots, g]))
                m = np.max([p[0] for p in parts], axis=0)
                w = [p[1] * np.exp(p[0] - m) for p in parts]
                lsum = np.sum(w, axis=0)
                o = np.sum([wi[:, None] * p[2] for wi, p in zip(w, parts)], axis=0) / lsum[:, None]
                out[r, j, g * G:(g + 1) * G, :] = o
    return out
