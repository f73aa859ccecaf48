"""fp64 oracle of the self-conditioning feed (test infrastructure; see the
package docstring).

Technical Report section 3.2, eq. 6: p0 = Softmax(L_t / tau_t) and the next
self-conditioning signal is FFW(p0 E), E the V x d token embedding.  This
function computes the contraction p0 E only; the feed-forward network, the
embedding scale and the add + RMSNorm around it are model side
("DiffusionGemma Explained", "Self-conditioning").

Rows that do not feed a next denoise step get zeros: the first decode step
sees all-zero self-conditioning ("DiffusionGemma Explained"), and the encoder
prefill / commit passes see it zeroed (vLLM blog, "Self-conditioning").
"""

from __future__ import annotations

import numpy as np


def softmax_rows(z, T):
    """p = softmax(z / T) per row in float64; rows that are invalid (NaN, +inf,
    all -inf) come back as all-zero rows."""
    z = np.asarray(z, dtype=np.float64)
    out = np.zeros_like(z)
    for i in range(z.shape[0]):
        row = z[i]
        if np.isnan(row).any() or np.isposinf(row).any() or not np.isfinite(row).any():
            continue
        y = row / T
        e = np.exp(y - np.max(y))
        out[i] = e / np.sum(e)
    return out


def selfcond_rows(z, T, E):
    """p0 E for the rows of ``z`` ([n, V]) at temperature ``T`` with the
    embedding ``E`` ([V, d], widened exactly to float64)."""
    P = softmax_rows(z, T)
    return P @ np.asarray(E, dtype=np.float64)


def selfcond(logits, temperature, E, feeds):
    """Full [B*C, d] output.  ``logits`` [B, C, V]; ``temperature`` [B];
    ``feeds`` [B] bool: rows that ran a denoise step and did not converge.
    Other rows are zero."""
    B, C, _ = logits.shape
    d = E.shape[1]
    out = np.zeros((B * C, d))
    for r in range(B):
        if feeds[r]:
            out[r * C:(r + 1) * C] = selfcond_rows(logits[r], float(temperature[r]), E)
    return out
