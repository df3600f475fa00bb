"""Mamba-2 linear recurrence (state-space duality form) oracle (test infrastructure only).

[Article] §6 ("Transfer: Nemotron, a Mamba hybrid architecture + NVFP4"): Mamba-2
is a linear recurrence; decode replays prefill's chunked arithmetic instead of
its own single-step recurrence, so both reach the same bits.  What the layer
computes is the plain recurrence below; the chunking is how the GPU orders it.

Per head h (heads share B and C within a group of H / G heads, as in Mamba-2):
    state_t = a_t * state_{t-1} + B_t x_t^T        state: [N, P], state_{-1} = 0
    y_t     = C_t^T state_t                        y: [P]
with a_t = exp(loga_t) (loga <= 0 per token and head), B_t, C_t in R^N, x_t in R^P.
The gate, the D skip term and the projections around the scan are elementwise
or GEMMs already covered elsewhere; this is the scan itself.

The oracle runs the recurrence one position after another in fp64: no chunks,
no blocking, no reordering.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own.
"""
from __future__ import annotations

import numpy as np


def ssd_scan(x, B, C, loga, n_groups: int = 1, state0=None):
    """x [T, H, P], B/C [T, G, N], loga [T, H] -> (y [T, H, P] fp64, final state [H, N, P] fp64)."""
    x = np.asarray(x, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    loga = np.asarray(loga, np.float64)
    T, H, P = x.shape
    N = B.shape[2]
    hpg = H // n_groups
    state = np.zeros((H, N, P)) if state0 is None else np.array(state0, np.float64)
    y = np.zeros((T, H, P))
    for t in range(T):
        for h in range(H):
            g = h // hpg
            state[h] = np.exp(loga[t, h]) * state[h] + np.outer(B[t, g], x[t, h])
            y[t, h] = C[t, g] @ state[h]
    return y, state
