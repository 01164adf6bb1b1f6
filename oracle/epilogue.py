"""fp64 output epilogue of the KDA layer -- TEST INFRASTRUCTURE ONLY (same rule as the rest
of ``oracle``: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs use it).

"Kimi K3.1 Pro 架构完全拆解", section 3.3 (full-rank output gate): the recurrent output of
each head is normalised by a head-wise RMSNorm and then gated channel by channel by the
sigmoid of an input-dependent projection, before the output projection W_o:

    y_t = W_o [ Sigmoid(W_g x_t) (.) RMSNorm(o~_t) ]

This module computes the bracket (the part that belongs to the recurrence's output stage):

    z_t = sigmoid(a_t) (.) gamma (.) o~_t / sqrt(mean_c(o~_t[c]^2) + eps)

per (token, head), with a_t = W_g x_t supplied as gate logits.  The page names the RMSNorm
without its weight or epsilon; the reading taken is the usual one -- a per-channel weight
gamma of length d shared by the heads (gamma = 1 when absent) and eps added to the mean
square inside the square root.
"""
from __future__ import annotations

import numpy as np


def sigmoid(a):
    a = np.asarray(a, np.float64)
    return 0.5 * (1.0 + np.tanh(0.5 * a))  # = 1 / (1 + e^-a), without overflow for large |a|


def gated_rmsnorm(o, gate_logits, gamma=None, eps=1e-5):
    """z = sigmoid(gate_logits) * gamma * o / sqrt(mean(o^2 over the last axis) + eps), fp64.

    ``o`` and ``gate_logits`` have the same shape (..., d); ``gamma`` has shape (d,)."""
    o = np.asarray(o, np.float64)
    a = np.asarray(gate_logits, np.float64)
    if a.shape != o.shape:
        raise ValueError("gate logits must have the shape of o")
    d = o.shape[-1]
    g = np.ones(d) if gamma is None else np.asarray(gamma, np.float64)
    if g.shape != (d,):
        raise ValueError("gamma must have shape (d,)")
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return sigmoid(a) * g * o / np.sqrt(ms + eps)
