"""Helpers shared by the GPU parity tests: host copies of device tensors, the oracle
run per (sequence, head) unit, and the error measures of the acceptance bar.

Tolerances (fixed by the acceptance bar for this path):
    prefill o      max|o - o_ref| / max|o_ref|            <= 1e-2   (bf16 output)
    prefill state  ||S - S_ref||_F / ||S_ref||_F          <= 1e-3   (final state, each checkpoint)
    decode o, S    max|x - x_ref| / max|x_ref|            <= 1e-4   (fp32 in and out)
    output stage y the o bar carried through the stage plus y's rounding (``y_bound``)
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle

O_TOL = 1e-2
S_TOL = 1e-3
DECODE_TOL = 1e-4


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def rel_max(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-300))


def rel_fro(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def y_bound(oref, gl, w, eps, omax):
    """Allowed |y - y_ref| per element of the output stage y = sigmoid(a) w o~ / rms(o~)
    ("Kimi K3.1 Pro 架构完全拆解" 3.3), for oracle rows ``oref`` [n, d] with gate logits ``gl``
    and weight ``w``; ``omax`` = max|o~_ref| over the whole checked tensor.  Returns (bound,
    y_ref).

    The o bar admits any o~' with |o~' - o~_ref| <= eps_o = O_TOL omax per element.  In a row
    of root mean square r (eps included) that moves y_c = s_c o~_c / r (s_c = sigmoid(a_c)
    |w_c|) by at most s_c eps_o (1 + |o~_c| / r) / (r - eps_o) -- exactly, not to first
    order: the numerator moves by at most eps_o and so does the root mean square (a norm).
    A row within 2 eps_o of zero is inside the o bar's noise and may take any value a
    normalised row can, |y_c| <= s_c sqrt(d).  y is then rounded to bf16 once (relative
    error at most 2^-8), and fp32 arithmetic adds 1e-6 max|y_ref|."""
    from oracle.epilogue import gated_rmsnorm, sigmoid
    oref = np.asarray(oref, np.float64)
    d = oref.shape[-1]
    eps_o = O_TOL * float(omax)
    s = sigmoid(gl) * np.abs(np.asarray(w, np.float64))
    r = np.sqrt(np.mean(oref ** 2, axis=-1, keepdims=True) + eps)
    with np.errstate(divide="ignore", invalid="ignore"):
        carried = s * eps_o * (1.0 + np.abs(oref) / r) / (r - eps_o)
    carried = np.where(r > 2 * eps_o, carried, s * np.sqrt(d))
    yr = gated_rmsnorm(oref, gl, w, eps)
    return carried + 2.0 ** -8 * np.abs(yr) + 1e-6 * np.abs(yr).max(), yr


def to_device(inp, device="cuda"):
    """Move a PrefillInputs / DecodeInputs to the device; index arrays become int32."""
    out = {}
    for name in ("q", "k", "v", "g", "beta", "S0"):
        t = getattr(inp, name)
        out[name] = None if t is None else t.to(device).contiguous()
    for name in ("cu_seqlens", "ckpt_off", "ckpt_pos", "n_commit"):
        t = getattr(inp, name, None)
        out[name] = None if t is None else t.to(device=device, dtype=torch.int32).contiguous()
    return out


def oracle_units(inp, units, o_stride=1, threads=None):
    """Run the oracle for each (seq, head) in ``units`` on that unit's rows alone.

    Returns {(seq, head): {"o": [len/o_stride, d] (rows 0, o_stride, ...), "S": [d, d],
    "ckpts": [n_ck, d, d] or None}} in fp64.  Units run concurrently (the oracle
    releases the GIL)."""
    cu = inp.cu_seqlens.cpu().numpy().astype(np.int64)
    off = None if inp.ckpt_off is None else inp.ckpt_off.cpu().numpy()
    pos = None if inp.ckpt_pos is None else inp.ckpt_pos.cpu().numpy()

    def one(unit):
        s, h = unit
        a, b = int(cu[s]), int(cu[s + 1])
        sl = lambda t: t[a:b, h:h + 1].contiguous()
        q, k, v = (bits(sl(getattr(inp, n))) for n in ("q", "k", "v"))
        g = host(sl(inp.g))
        beta = host(inp.beta[a:b, h:h + 1].contiguous())
        S0 = None if inp.S0 is None else host(inp.S0[s:s + 1, h:h + 1].contiguous())
        co = cp = None
        if off is not None:
            p = pos[off[s]:off[s + 1]].astype(np.int32)
            co = np.array([0, p.shape[0]], np.int32)
            cp = p
        rows = None
        if o_stride > 1:
            rows = np.arange(0, b - a, o_stride, dtype=np.int64)
        r = oracle.prefill(q, k, v, g, beta, np.array([0, b - a], np.int32), S_in=S0, ckpt_off=co,
                           ckpt_pos=cp, o_rows=rows, n_threads=1)
        return unit, {"o": r["o"][:, 0], "S": r["S_out"][0, 0],
                      "ckpts": None if r["ckpts"] is None else r["ckpts"][:, 0]}

    n = threads or max(1, min(len(units), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        return dict(ex.map(one, units))
