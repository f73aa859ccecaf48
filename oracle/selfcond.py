"""fp64 oracle of the self-conditioning feed (test infrastructure; see the
package docstring).

Technical Report section 3.2, eq. 6: p0 = Softmax(L_t / tau_t) and the next
self-conditioning signal is FFW(p0 E), E the V x d token embedding.  This
module computes the contraction p0 E, optionally times the embedding scale
("The Annotated DiffusionGemma", the model's forward: the probabilities times
W_embed, times embed_scale) and with p0 taken over softcapped logits ("Logit
Softcapping" on the same page).  The feed-forward network and the add +
RMSNorm around it are model side ("DiffusionGemma Explained",
"Self-conditioning").

Rows that do not feed a next denoise step get zeros: the first decode step
sees all-zero self-conditioning ("DiffusionGemma Explained"), and the encoder
prefill / commit passes see it zeroed (vLLM blog, "Self-conditioning").
"""

from __future__ import annotations

import numpy as np

from oracle.sampler import softcap as _softcap


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


def selfcond_rows(z, T, E, cap=0.0, scale=0.0):
    """p0 E for the rows of ``z`` ([n, V]) at temperature ``T`` with the
    embedding ``E`` ([V, d], widened exactly to float64).  ``cap`` > 0
    softcaps the logits first; ``scale`` multiplies the result (0 means 1)."""
    P = softmax_rows(_softcap(z, cap), T)
    out = P @ np.asarray(E, dtype=np.float64)
    return out * scale if scale != 0 else out


def selfcond(logits, temperature, E, feeds, cap=0.0, scale=0.0):
    """Full [B*C, d] output.  ``logits`` [B, C, V]; ``temperature`` [B];
    ``feeds`` [B] bool: rows that ran a denoise step and did not converge.
    Other rows are zero.  ``cap`` and ``scale`` as in ``selfcond_rows``."""
    B, C, _ = logits.shape
    d = E.shape[1]
    out = np.zeros((B * C, d))
    for r in range(B):
        if feeds[r]:
            out[r * C:(r + 1) * C] = selfcond_rows(logits[r], float(temperature[r]), E, cap, scale)
    return out
