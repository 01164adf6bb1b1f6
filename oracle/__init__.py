"""fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence.

TEST INFRASTRUCTURE ONLY: the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the library under
``kimi_delta_attention_prefill_gb300`` never does, and this package never imports it.

Contents
--------
``prefill`` / ``decode``
    ctypes front-end of ``kda_oracle.c``: the per-token recurrence of
    "Kimi K3.1 Pro 架构完全拆解" section 3.1, in fp64, threads over (sequence, head).
``chunked``
    an fp64 numpy restatement of the chunk-level matrix form ("FlashKDA 演算法",
    section 6 of the SemiAnalysis translation) -- used only to show that the chunk
    algebra reproduces the per-token recurrence.
``segments``
    the segment algebra of "部署 Kimi K3 ..." section 2 (cumulative transition M,
    zero-start state S~, combine, entry state S = S~ + M S_in).
``epilogue``
    the output stage of "Kimi K3.1 Pro 架构完全拆解" section 3.3: head-wise RMSNorm of the
    recurrent output, gated channel by channel by the sigmoid of supplied gate logits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` (plain C, -O2, no fast-math) into ``libkda_oracle.so``."""
    hdr = os.path.join(_HERE, "kda_oracle.h")
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(hdr))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("qkv_is_f32", ctypes.c_int),
        ("g", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("S_in", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p),
        ("n_seq", ctypes.c_int), ("H", ctypes.c_int), ("d", ctypes.c_int),
        ("ckpt_off", ctypes.c_void_p), ("ckpt_pos", ctypes.c_void_p),
        ("units", ctypes.c_void_p), ("n_units", ctypes.c_int64),
        ("o", ctypes.c_void_p), ("o_rows", ctypes.c_void_p), ("n_o_rows", ctypes.c_int64),
        ("S_out", ctypes.c_void_p), ("ckpts", ctypes.c_void_p),
        ("n_threads", ctypes.c_int),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.kda_ref_run.restype = ctypes.c_int
            lib.kda_ref_run.argtypes = [ctypes.POINTER(_Args), ctypes.POINTER(ctypes.c_int)]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _qkv(x):
    """bf16 bit patterns (uint16 / int16) pass through; anything else becomes float32."""
    x = np.asarray(x)
    if x.dtype in (np.uint16, np.int16):
        return np.ascontiguousarray(x.view(np.uint16)), 0
    return np.ascontiguousarray(x, dtype=np.float32), 1


class OracleError(RuntimeError):
    pass


def prefill(q, k, v, g, beta, cu_seqlens, S_in=None, ckpt_off=None, ckpt_pos=None,
            units=None, o_rows=None, want_o=True, n_threads=0):
    """Run the fp64 per-token recurrence over packed sequences.

    Shapes: q, k, v, g ``[T_tot, H, d]`` (q/k/v as bf16 bits or float32), beta
    ``[T_tot, H]``, S_in ``[N, H, d, d]`` or None, cu_seqlens ``[N+1]``.
    ``units`` restricts the work to the listed ``seq * H + head`` indices; ``o_rows``
    keeps outputs for the listed packed rows only (ascending).

    Returns a dict with ``o`` (fp64, ``[T_tot or len(o_rows), H, d]`` or None),
    ``S_out`` ``[N, H, d, d]``, ``ckpts`` ``[n_ckpt, H, d, d]`` (or None) and
    ``threads``.  Entries of units that were not requested are left at zero.
    """
    lib = _load()
    qa, f32 = _qkv(q)
    ka, f32k = _qkv(k)
    va, f32v = _qkv(v)
    if not (f32 == f32k == f32v):
        raise OracleError("q, k, v must share one element type")
    T_tot, H, d = qa.shape
    ga = _c(g, np.float32)
    ba = _c(beta, np.float32)
    cu = _c(cu_seqlens, np.int32)
    n_seq = cu.shape[0] - 1
    s0 = _c(S_in, np.float32)
    co = _c(ckpt_off, np.int32)
    cp = _c(ckpt_pos, np.int32)
    un = _c(units, np.int64)
    orow = _c(o_rows, np.int64)
    n_rows = T_tot if orow is None else orow.shape[0]
    o = np.zeros((n_rows, H, d), np.float64) if want_o else None
    S_out = np.zeros((n_seq, H, d, d), np.float64)
    n_ck = 0 if co is None else int(co[-1])
    ckpts = np.zeros((n_ck, H, d, d), np.float64) if co is not None else None
    args = _Args(
        q=_ptr(qa), k=_ptr(ka), v=_ptr(va), qkv_is_f32=f32, g=_ptr(ga), beta=_ptr(ba),
        S_in=_ptr(s0), cu_seqlens=_ptr(cu), n_seq=n_seq, H=H, d=d,
        ckpt_off=_ptr(co), ckpt_pos=_ptr(cp),
        units=_ptr(un), n_units=0 if un is None else un.shape[0],
        o=_ptr(o), o_rows=_ptr(orow), n_o_rows=0 if orow is None else orow.shape[0],
        S_out=_ptr(S_out), ckpts=_ptr(ckpts) if ckpts is not None and n_ck > 0 else None,
        n_threads=int(n_threads))
    used = ctypes.c_int(0)
    st = lib.kda_ref_run(ctypes.byref(args), ctypes.byref(used))
    if st != 0:
        raise OracleError(f"kda_ref_run failed with status {st}")
    return {"o": o, "S_out": S_out, "ckpts": ckpts, "threads": used.value}


def decode(q, k, v, g, beta, S_state, n_commit=None, n_threads=0):
    """Multi-token decode / verify in fp64.

    q, k, v, g ``[B, n_tok, H, d]``; beta ``[B, n_tok, H]``; S_state ``[B, H, d, d]``;
    n_commit ``[B]`` in ``[0, n_tok]`` or None (= n_tok).  Each batch entry is a
    sequence of n_tok tokens starting from its own state; the outputs of all n_tok
    tokens are returned, and the committed state is the state after n_commit tokens
    ("部署 Kimi K3 ..." section 4: replay the accepted prefix, write back its state).
    Returns ``{"o": [B, n_tok, H, d], "S": [B, H, d, d]}`` in fp64.
    """
    qa, _ = _qkv(q)
    B, n_tok, H, d = qa.shape
    flat = lambda x: np.asarray(x).reshape((B * n_tok,) + np.asarray(x).shape[2:])
    cu = np.arange(B + 1, dtype=np.int32) * n_tok
    nc = np.full(B, n_tok, np.int32) if n_commit is None else np.asarray(n_commit, np.int32)
    if nc.shape != (B,) or (nc < 0).any() or (nc > n_tok).any():
        raise OracleError("n_commit must be [B] with entries in [0, n_tok]")
    off = np.zeros(B + 1, np.int32)
    off[1:] = np.cumsum(nc > 0)
    pos = nc[nc > 0].astype(np.int32)
    r = prefill(flat(q), flat(k), flat(v), flat(g), flat(beta), cu, S_in=S_state,
                ckpt_off=off, ckpt_pos=pos, n_threads=n_threads)
    S = np.asarray(S_state, np.float64).copy()
    idx = np.nonzero(nc > 0)[0]
    if idx.size:
        S[idx] = r["ckpts"]
    return {"o": r["o"].reshape(B, n_tok, H, d), "S": S}
