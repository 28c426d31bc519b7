"""Trie-constrained beam expansion (oracle side).

What one expansion step computes, following "Generative recommendation design"
§4.1.1 (every beam expands top_k candidates, then beam_width beams are chosen
from the beam_width x top_k pool), §4.3 (invalid item paths are filtered before
they become candidates), §6 (beam search, then cache selection after the
reorder) and "Deploying FlashRec" (temperature 0 = deterministic top-k; the
returned sequence score is the cumulative log-probability):

1. ``lse_b = log sum_v exp(logit[b, v])`` over the full vocabulary, in float64.
2. Candidates of beam b: the children of its trie node at level ``level``
   (token = token_base[level] + code), or every token with no trie.
3. Candidate score ``s = fl32(cum_b + fl32(logit - lse32_b))``: float32
   round-to-nearest-even, no fused multiply-add.  ``lse32_b`` is the float32
   rounding of ``lse_b`` unless the caller passes the float32 normaliser to use
   (so that both sides take the integer decisions on identical float32 scores).
4. Per beam: full sort by (s desc, token asc), keep the first min(top_k, n).
5. Per request: full sort of the pool by (s desc, parent beam asc, token asc),
   keep the first beam_width.  n_live' = min(beam_width, pool size).
6. Outputs in rank order j: token, parent beam, cumulative score s, child node;
   slot row j = the parent's slot row up to ``step`` - 1, then ``step*W + j``
   (the slot of the token just chosen; KV is never copied).  Rows j >= n_live'
   hold token = parent = node = -1 and cum = -inf; their slot rows are
   unspecified.

Step 0 starts from one live beam per request (the prefill row, cum = 0).

With temperature > 0 (Gumbel top-k, "Deploying FlashRec" serving
parameters), steps 4 and 5 order by the noisy key of ``oracle.gumbel``
(fl32(fl32(s * inv_tau) + g), ties as above) instead of s; the returned
cumulative score stays s, without the noise.
"""
import numpy as np

from oracle import gumbel as _gumbel

F32 = np.float32


def lse64(row) -> float:
    """Float64 log-sum-exp of one logits row (max-subtracted)."""
    x = np.asarray(row, dtype=np.float64)
    m = x.max()
    return float(m + np.log(np.exp(x - m).sum()))


def candidates(trie, token_base, level, node, V):
    """(tokens int64, child nodes int64) a beam at ``node`` may extend with."""
    if trie is None:
        return np.arange(V, dtype=np.int64), np.full(V, -1, dtype=np.int64)
    codes, kids = trie.children(level, node)
    return int(token_base[level]) + codes.astype(np.int64), kids.astype(np.int64)


def candidate_scores(x_f32, cum_f32, lse_f32):
    """fl32(cum + fl32(x - lse)) with float32 round-to-nearest-even steps."""
    lp = (np.asarray(x_f32, dtype=F32) - F32(lse_f32)).astype(F32)
    return (F32(cum_f32) + lp).astype(F32)


def beam_select(logits, cum, node, n_live, slot_in, trie, token_base, level, step,
                W, K, lse32=None, temperature=0.0, seed=0):
    """One expansion step for every request.

    logits [R, >=n_live, V] float32; cum [R, W] float32; node [R, W] int;
    n_live [R]; slot_in [R, W, T] int32.  Returns a dict of numpy arrays:
    tokens, parents, cum_out, node_out [R, W]; n_live_out [R]; slot_out
    [R, W, T]; lse64 [R, W] (NaN for dead rows).  temperature > 0: Gumbel
    top-k with the counter-based noise of ``oracle.gumbel`` under ``seed``.
    """
    gumbel = temperature > 0
    itau = _gumbel.inv_tau(temperature) if gumbel else None
    logits = np.asarray(logits)
    R, V = logits.shape[0], logits.shape[2]
    T = slot_in.shape[2]
    tokens = np.full((R, W), -1, dtype=np.int32)
    parents = np.full((R, W), -1, dtype=np.int32)
    cum_out = np.full((R, W), -np.inf, dtype=F32)
    node_out = np.full((R, W), -1, dtype=np.int64)
    n_live_out = np.zeros(R, dtype=np.int32)
    slot_out = np.full((R, W, T), -1, dtype=np.int32)
    lse_all = np.full((R, W), np.nan)
    for r in range(R):
        ps, pb, pt, pc, pk = [], [], [], [], []
        for b in range(int(n_live[r])):
            row = logits[r, b]
            lse_all[r, b] = lse64(row)
            l32 = F32(lse_all[r, b]) if lse32 is None else F32(lse32[r, b])
            tok, kid = candidates(trie, token_base, level, int(node[r, b]), V)
            s = candidate_scores(row[tok], cum[r, b], l32)
            key = (_gumbel.ordering_keys(s, _gumbel.gumbel(seed, r, step, b, tok), itau) if gumbel else s)
            order = np.lexsort((tok, -key.astype(np.float64)))[: min(K, len(tok))]
            ps.append(s[order]); pb.append(np.full(len(order), b)); pt.append(tok[order]); pc.append(kid[order])
            pk.append(key[order])
        if not ps:
            continue
        s, b, t, c, key = (np.concatenate(a) for a in (ps, pb, pt, pc, pk))
        order = np.lexsort((t, b, -key.astype(np.float64)))[:W]
        n = len(order)
        n_live_out[r] = n
        tokens[r, :n] = t[order]
        parents[r, :n] = b[order]
        cum_out[r, :n] = s[order]
        node_out[r, :n] = c[order]
        for j in range(n):
            slot_out[r, j, :step] = slot_in[r, parents[r, j], :step]
            slot_out[r, j, step] = step * W + j
    return dict(tokens=tokens, parents=parents, cum_out=cum_out, node_out=node_out,
                n_live_out=n_live_out, slot_out=slot_out, lse64=lse_all)


def beam_select_bruteforce(logits, cum, node, n_live, trie, token_base, level, W, K,
                           lse32=None, temperature=0.0, seed=0, step=0):
    """Single-pass restatement used only to pin ``beam_select`` on tiny inputs.

    Enumerates every (beam, token) pair of the whole beam x vocab grid, drops the
    pairs the trie forbids, orders all of them by (s desc, beam asc, token asc)
    and walks that order keeping at most top_k per beam, stopping at beam_width.
    With temperature > 0 the order is by the noisy key instead (the noise of
    each pair drawn on its own).  Plain Python loops: tiny sizes only.
    """
    R, V = logits.shape[0], logits.shape[2]
    out = []
    for r in range(R):
        allc = []
        for b in range(int(n_live[r])):
            l32 = F32(lse64(logits[r, b])) if lse32 is None else F32(lse32[r, b])
            if trie is None:
                allowed = {v: -1 for v in range(V)}
            else:
                codes, kids = trie.children(level, int(node[r, b]))
                allowed = {int(token_base[level]) + int(c): int(k) for c, k in zip(codes, kids)}
            for v in range(V):
                if v in allowed:
                    s = F32(F32(cum[r, b]) + F32(F32(logits[r, b, v]) - l32))
                    key = s
                    if temperature > 0:
                        g = _gumbel.gumbel(seed, r, step, b, np.array([v]))[0]
                        key = F32(F32(s * _gumbel.inv_tau(temperature)) + g)
                    allc.append((-float(key), b, v, allowed[v], s))
        allc.sort()
        taken, per_beam = [], {}
        for neg_s, b, v, kid, s in allc:
            if per_beam.get(b, 0) >= K:
                continue
            per_beam[b] = per_beam.get(b, 0) + 1
            taken.append((v, b, s, kid))
            if len(taken) == W:
                break
        out.append(taken)
    return out
