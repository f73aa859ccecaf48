"""Forward-process transition row of uniform-state diffusion (test
infrastructure; see the package docstring).

Technical Report section 2.1.1, eq. 1: per coordinate,
P(x_t = v | x_0) = kappa_t * delta(v, x_0) + (1 - kappa_t) / V.
Used only as an invariant of the oracle (a distribution over V tokens).
"""

from __future__ import annotations

import numpy as np


def transition_row(x0: int, kappa: float, V: int) -> np.ndarray:
    row = np.full(V, (1.0 - kappa) / V)
    row[x0] += kappa
    return row
