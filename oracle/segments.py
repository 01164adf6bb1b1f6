"""Segment algebra for splitting one sequence into independently computed pieces
(test infrastructure only).

Source: "部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra 全景", section 2 (the KCP
mathematics) and section 1.2 (the same decomposition applied across the SMs of one GPU):

    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t)              per-token transition
    M   = M_T ... M_1                                         cumulative transition
    S~  = state the segment produces from a zero entry state
    S   = S~ + M S_in                                         exit state for entry S_in

Pieces compose associatively: (M2, S~2) o (M1, S~1) = (M2 M1, S~2 + M2 S~1), so the
entry state of every piece follows from an inclusive prefix scan of the preceding pairs.
The transition here is the literal matrix product of the page's definition, in fp64.
"""
from __future__ import annotations

import numpy as np


def transition(k, g, beta):
    """Cumulative transition of one segment: k, g ``[T, d]`` (fp64-able), beta ``[T]``."""
    k = np.asarray(k, np.float64)
    g = np.asarray(g, np.float64)
    beta = np.asarray(beta, np.float64)
    T, d = k.shape
    M = np.eye(d)
    I = np.eye(d)
    for t in range(T):
        Mt = (I - beta[t] * np.outer(k[t], k[t])) @ np.diag(np.exp(g[t]))
        M = Mt @ M
    return M


def combine(first, second):
    """Pair for ``first`` followed by ``second``; each pair is (M, S~)."""
    M1, S1 = first
    M2, S2 = second
    return M2 @ M1, S2 + M2 @ S1


def exit_state(pair, S_in):
    M, St = pair
    return St + M @ np.asarray(S_in, np.float64)


def entry_states(pairs, S_in):
    """Entry state of each segment given the pairs of all segments, in order."""
    out = []
    S = np.asarray(S_in, np.float64)
    for p in pairs:
        out.append(S)
        S = exit_state(p, S)
    return out, S
