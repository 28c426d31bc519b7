"""LM head and its log-sum-exp (oracle side; test infrastructure).

The step before the selection ("Generative recommendation design" §4.3
filters invalid items before they become candidates): logits = hidden x W^T
over the whole vocabulary, then each row's ln sum_v exp(logit).  Computed in
float64 from the bf16 inputs (every bf16 value and every product of two is
exact in float64; the sums are float64).
"""
import numpy as np

from oracle import select as osel


def logits64(hidden_f64, weight_f64, rows=None):
    """float64 logits [len(rows), V] for the chosen rows (all by default)."""
    h = hidden_f64 if rows is None else hidden_f64[rows]
    return h @ weight_f64.T


def lse_rows(hidden_f64, weight_f64, rows=None):
    lg = logits64(hidden_f64, weight_f64, rows)
    return np.array([osel.lse64(x) for x in lg]), lg
