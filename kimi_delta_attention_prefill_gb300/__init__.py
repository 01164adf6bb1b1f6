"""GB300-native Kimi Delta Attention (KDA): chunkwise prefill and decode / verify.

Python binding of the C ABI in ``include/kda.h``: argument marshalling only.  Every
step of the computation runs in the CUDA kernels of ``libkda.so`` (sm_103a); there is
no CPU or PyTorch fallback, and a missing library raises ``KdaLibraryError``.

Functions mirror the C entry points: :func:`prefill` (``kda_prefill``, or
``kda_prefill_gated`` when gate logits are given), :func:`prefill_paged`
(``kda_prefill_paged``), :func:`prefill_host` (``kda_prefill_host``, host buffers),
:func:`decode` (``kda_decode``), :func:`decode_paged` (``kda_decode_paged``),
:func:`decode_fused` (``kda_decode_fused``), :func:`prefill_pairs` (``kda_prefill_pairs``),
:func:`combine_pairs` (``kda_combine_pairs``), :func:`prefill_noalloc`
(``kda_prefill_noalloc``), the workspace-size queries, and :func:`status_string`
(``kda_status_string``).  The cross-device split's exchange is in :mod:`.kcp`.  Tensors are torch CUDA tensors (pinned
host tensors for :func:`prefill_host`); the launch goes to the current torch stream
unless ``stream`` is given.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")
HEAD_DIM = 128
CHUNK = 64
MAX_DECODE_TOKENS = 4

_lib = None
_lock = threading.Lock()

_c_int, _c_i64, _c_sz, _vp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p


class KdaLibraryError(RuntimeError):
    """The compiled CUDA library is missing or cannot be loaded."""


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


def library():
    """Load ``libkda.so`` (built by ``kimi_delta_attention_prefill_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise KdaLibraryError(
                    f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
            try:
                lib = ctypes.CDLL(LIB_PATH)
            except OSError as e:  # pragma: no cover - depends on the host
                raise KdaLibraryError(f"cannot load {LIB_PATH}: {e}") from e
            lib.kda_status_string.restype = ctypes.c_char_p
            lib.kda_status_string.argtypes = [_c_int]
            lib.kda_version.restype = _c_int
            lib.kda_version.argtypes = []
            lib.kda_decode.restype = _c_int
            lib.kda_decode.argtypes = [_vp] * 8 + [_c_int] * 4 + [_vp, _vp]
            lib.kda_prefill_workspace_size.restype = _c_sz
            lib.kda_prefill_workspace_size.argtypes = [_c_int, _c_int, _c_int, _c_i64, _c_int]
            lib.kda_prefill.restype = _c_int
            lib.kda_prefill.argtypes = ([_vp] * 7 + [_c_int, _c_i64] + [_vp, _vp, _c_i64] + [_vp] * 3 +
                                        [_c_int, _c_int, _c_int, _vp, _c_sz, _vp, _vp])
            lib.kda_prefill_gated.restype = _c_int
            lib.kda_prefill_gated.argtypes = ([_vp] * 7 + [ctypes.c_float] + [_vp, _vp] + [_c_int, _c_i64] +
                                              [_vp, _vp, _c_i64] + [_vp] * 3 +
                                              [_c_int, _c_int, _c_int, _vp, _c_sz, _vp, _vp])
            lib.kda_prefill_paged_workspace_size.restype = _c_sz
            lib.kda_prefill_paged_workspace_size.argtypes = [_c_int, _c_int, _c_int, _c_i64, _c_int, _c_i64]
            lib.kda_prefill_paged.restype = _c_int
            lib.kda_prefill_paged.argtypes = ([_vp] * 7 + [ctypes.c_float] + [_vp, _c_i64, _vp, _vp, _vp] +
                                              [_c_int, _c_i64, _vp, _vp, _c_i64, _vp, _vp] +
                                              [_c_int, _c_int, _c_int, _vp, _c_sz, _vp, _vp])
            lib.kda_decode_paged_workspace_size.restype = _c_sz
            lib.kda_decode_paged_workspace_size.argtypes = [_c_i64]
            lib.kda_decode_paged.restype = _c_int
            lib.kda_decode_paged.argtypes = ([_vp] * 6 + [_c_i64] + [_vp] * 4 + [_c_int] * 4 +
                                             [_vp, _c_sz, _vp, _vp])
            lib.kda_decode_fused.restype = _c_int
            lib.kda_decode_fused.argtypes = ([_vp] * 5 + [_c_int, _c_int] + [_vp, _vp, ctypes.c_float] + [_vp] * 3 +
                                             [ctypes.c_float] + [_vp] * 3 + [_c_int] * 4 + [_vp, _vp])
            lib.kda_prefill_host_workspace_size.restype = _c_sz
            lib.kda_prefill_host_workspace_size.argtypes = [_c_int, _c_int, _c_int, _c_i64, _c_i64]
            lib.kda_prefill_host.restype = _c_int
            lib.kda_prefill_host.argtypes = ([_vp] * 7 + [_c_int, _c_i64, _vp, _vp, _c_int, _c_int, _c_i64] +
                                             [_vp, _c_sz, _vp, _vp])
            lib.kda_prefill_host_blocks.restype = _c_int
            lib.kda_prefill_host_blocks.argtypes = [_vp, _c_int, _c_i64, _c_i64, _vp, _c_int]
            if hasattr(lib, "kda_debug_stall_next_prefill"):  # diagnostic hook (tests)
                lib.kda_debug_stall_next_prefill.restype = None
                lib.kda_debug_stall_next_prefill.argtypes = [_c_int]
            lib.kda_prefill_pairs.restype = _c_int
            lib.kda_prefill_pairs.argtypes = [_vp] * 6 + [_c_int, _c_i64, _vp, _vp, _c_int, _c_int, _vp, _vp]
            lib.kda_combine_pairs.restype = _c_int
            lib.kda_combine_pairs.argtypes = [_vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _vp]
            lib.kda_prefill_noalloc.restype = _c_int
            lib.kda_prefill_noalloc.argtypes = ([_vp] * 7 + [_c_int, _c_i64] + [_vp, _vp, _c_i64] + [_vp] * 3 +
                                                [_c_int, _c_int, _c_int, _vp, _vp])
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().kda_status_string(int(status)).decode()


def version() -> int:
    return library().kda_version()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def decode(q, k, v, g, beta, S_state, n_commit=None, o=None, dev_status=None, stream=None):
    """One decode (n_tok = 1) or verify (n_tok <= 4) step; updates ``S_state`` in place.

    q, k, v ``[B, n_tok, H, 128]`` bf16; g ``[B, n_tok, H, 128]`` fp32; beta
    ``[B, n_tok, H]`` fp32; S_state ``[B, H, 128, 128]`` fp32; n_commit ``[B]`` int32 or
    None.  Returns o ``[B, n_tok, H, 128]`` fp32.
    """
    B, n_tok, H, d = q.shape
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape)
    _need(beta, "beta", torch.float32, (B, n_tok, H))
    _need(S_state, "S_state", torch.float32, (B, H, d, d))
    if n_commit is not None:
        _need(n_commit, "n_commit", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, n_tok, H, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, n_tok, H, d))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    st = library().kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S_state), _ptr(n_commit),
                              _ptr(o), B, n_tok, H, d, _ptr(dev_status), _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_decode")
    return o


def decode_fused(qp, kp, vp, conv_w, conv_cache, z, a_log, b, S_state, n_commit=None, conv_act="none",
                 g_min=-5.0, gate=None, norm_weight=None, eps=1e-5, o=None, dev_status=None, stream=None):
    """A decode / verify step from projected inputs (``kda_decode_fused``): short causal
    convolution (``conv_w`` ``[3, H, 128, W]``, ``conv_cache`` ``[B, H, 3, W-1, 128]``, updated
    in place to the committed tokens), q / k L2 normalisation, alpha = exp(g_min
    sigmoid(e^a_log z)), beta = sigmoid(b), the recurrence on ``S_state`` (in place) and, with
    ``gate``, the output stage.  qp, kp, vp ``[B, n_tok, H, 128]`` bf16; z fp32 of the same
    shape; a_log ``[H]``; b ``[B, n_tok, H]``.  Returns o ``[B, n_tok, H, 128]`` fp32."""
    B, n_tok, H, d = qp.shape
    _need(qp, "qp", torch.bfloat16)
    _need(kp, "kp", torch.bfloat16, qp.shape)
    _need(vp, "vp", torch.bfloat16, qp.shape)
    _need(conv_w, "conv_w", torch.float32)
    if conv_w.dim() != 4 or tuple(conv_w.shape[:3]) != (3, H, d):
        raise ValueError(f"conv_w must have shape [3, {H}, {d}, W], got {tuple(conv_w.shape)}")
    W = conv_w.shape[3]
    if W > 1:
        _need(conv_cache, "conv_cache", torch.float32, (B, H, 3, W - 1, d))
    _need(z, "z", torch.float32, qp.shape)
    _need(a_log, "a_log", torch.float32, (H,))
    _need(b, "b", torch.float32, (B, n_tok, H))
    _need(S_state, "S_state", torch.float32, (B, H, d, d))
    if n_commit is not None:
        _need(n_commit, "n_commit", torch.int32, (B,))
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, qp.shape)
        if norm_weight is not None:
            _need(norm_weight, "norm_weight", torch.float32, (d,))
    if o is None:
        o = torch.empty((B, n_tok, H, d), dtype=torch.float32, device=qp.device)
    _need(o, "o", torch.float32, (B, n_tok, H, d))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    act = {"none": 0, "silu": 1}[conv_act]
    st = library().kda_decode_fused(_ptr(qp), _ptr(kp), _ptr(vp), _ptr(conv_w), _ptr(conv_cache) if W > 1 else None,
                                    W, act, _ptr(z), _ptr(a_log), float(g_min), _ptr(b), _ptr(gate),
                                    _ptr(norm_weight), float(eps), _ptr(S_state), _ptr(n_commit), _ptr(o), B, n_tok,
                                    H, d, _ptr(dev_status), _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_decode_fused")
    return o


def prefill_workspace_size(n_seq, H, total_tokens, n_segments=0, d=HEAD_DIM) -> int:
    return int(library().kda_prefill_workspace_size(int(n_seq), int(H), int(d), int(total_tokens),
                                                    int(n_segments)))


def prefill(q, k, v, g, beta, cu_seqlens, S_in=None, ckpt_off=None, ckpt_pos=None, o=None, S_out=None,
            ckpts=None, n_segments=0, workspace=None, dev_status=None, stream=None, gate=None,
            norm_weight=None, eps=1e-5):
    """Chunkwise prefill over packed sequences.

    q, k, v ``[T, H, 128]`` bf16; g ``[T, H, 128]`` fp32; beta ``[T, H]`` fp32;
    cu_seqlens ``[N+1]`` int32 (device); S_in ``[N, H, 128, 128]`` fp32 or None;
    ckpt_off ``[N+1]`` / ckpt_pos ``[n_ckpt]`` int32 (device) or None.
    With ``gate`` (``[T, H, 128]`` bf16 gate logits) the output stage is fused
    (``kda_prefill_gated``): the returned ``o`` holds
    ``sigmoid(gate) * norm_weight * o~ / sqrt(mean(o~^2) + eps)`` (``norm_weight`` ``[128]``
    fp32 or None for ones).
    Returns ``(o, S_out, ckpts)``.
    """
    T, H, d = q.shape
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape)
    _need(beta, "beta", torch.float32, (T, H))
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    n_seq = cu_seqlens.shape[0] - 1
    if S_in is not None:
        _need(S_in, "S_in", torch.float32, (n_seq, H, d, d))
    n_ckpt = 0
    if ckpt_off is not None:
        _need(ckpt_off, "ckpt_off", torch.int32, (n_seq + 1,))
        _need(ckpt_pos, "ckpt_pos", torch.int32)
        n_ckpt = ckpt_pos.shape[0]
        if ckpts is None:
            ckpts = torch.empty((n_ckpt, H, d, d), dtype=torch.float32, device=q.device)
        _need(ckpts, "ckpts", torch.float32, (n_ckpt, H, d, d))
    if o is None:
        o = torch.empty((T, H, d), dtype=torch.bfloat16, device=q.device)
    _need(o, "o", torch.bfloat16, (T, H, d))
    if S_out is None:
        S_out = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=q.device)
    _need(S_out, "S_out", torch.float32, (n_seq, H, d, d))
    ws_need = prefill_workspace_size(n_seq, H, T, n_segments, d)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    if gate is None:
        st = library().kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S_in), _ptr(cu_seqlens),
                                   n_seq, T, _ptr(ckpt_off), _ptr(ckpt_pos), n_ckpt, _ptr(o), _ptr(S_out),
                                   _ptr(ckpts), H, d, int(n_segments), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                   _stream_handle(stream))
        if st != 0:
            raise KdaError(st, "kda_prefill")
        return o, S_out, ckpts
    _need(gate, "gate", torch.bfloat16, q.shape)
    if norm_weight is not None:
        _need(norm_weight, "norm_weight", torch.float32, (d,))
    st = library().kda_prefill_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(gate), _ptr(norm_weight),
                                     float(eps), _ptr(S_in), _ptr(cu_seqlens), n_seq, T, _ptr(ckpt_off),
                                     _ptr(ckpt_pos), n_ckpt, _ptr(o), _ptr(S_out), _ptr(ckpts), H, d,
                                     int(n_segments), _ptr(workspace), ws_bytes, _ptr(dev_status),
                                     _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_prefill_gated")
    return o, S_out, ckpts


def _pool(state_pool, d):
    _need(state_pool, "state_pool", torch.float32)
    if state_pool.dim() != 3 or tuple(state_pool.shape[1:]) != (d, d):
        raise ValueError(f"state_pool must have shape [n_pages, {d}, {d}], got {tuple(state_pool.shape)}")
    return state_pool.shape[0]


def _table(t, name, n):
    if t is not None:
        _need(t, name, torch.int32, (n,))
    return t


def prefill_paged_workspace_size(n_seq, H, total_tokens, n_pages, n_segments=0, d=HEAD_DIM) -> int:
    return int(library().kda_prefill_paged_workspace_size(int(n_seq), int(H), int(d), int(total_tokens),
                                                          int(n_segments), int(n_pages)))


def prefill_paged(q, k, v, g, beta, cu_seqlens, state_pool, s_in_page=None, s_out_page=None, ckpt_off=None,
                  ckpt_pos=None, ckpt_page=None, o=None, n_segments=0, workspace=None, dev_status=None,
                  stream=None, gate=None, norm_weight=None, eps=1e-5):
    """:func:`prefill` with every state in a page pool (``kda_prefill_paged``).

    state_pool ``[n_pages, 128, 128]`` fp32; s_in_page / s_out_page ``[N * H]`` int32
    (entry ``seq * H + h``; -1 = zeros / not written; None = all zeros / none); ckpt_page
    ``[n_ckpt * H]`` int32 (entry ``j * H + h``).  A call never writes a page it reads
    (except a unit's own final state in place) and writes each page once; a violation
    writes nothing and sets ``dev_status`` to KDA_ERR_DEVICE_CHECK.  Returns ``o``.
    """
    T, H, d = q.shape
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape)
    _need(beta, "beta", torch.float32, (T, H))
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    n_seq = cu_seqlens.shape[0] - 1
    n_pages = _pool(state_pool, d)
    _table(s_in_page, "s_in_page", n_seq * H)
    _table(s_out_page, "s_out_page", n_seq * H)
    n_ckpt = 0
    if ckpt_off is not None:
        _need(ckpt_off, "ckpt_off", torch.int32, (n_seq + 1,))
        _need(ckpt_pos, "ckpt_pos", torch.int32)
        n_ckpt = ckpt_pos.shape[0]
        _table(ckpt_page, "ckpt_page", n_ckpt * H)
    if o is None:
        o = torch.empty((T, H, d), dtype=torch.bfloat16, device=q.device)
    _need(o, "o", torch.bfloat16, (T, H, d))
    if gate is not None:
        _need(gate, "gate", torch.bfloat16, q.shape)
        if norm_weight is not None:
            _need(norm_weight, "norm_weight", torch.float32, (d,))
    if workspace is None:
        need = prefill_paged_workspace_size(n_seq, H, T, n_pages, n_segments, d)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    st = library().kda_prefill_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(gate), _ptr(norm_weight),
                                     float(eps), _ptr(state_pool), n_pages, _ptr(s_in_page), _ptr(s_out_page),
                                     _ptr(cu_seqlens), n_seq, T, _ptr(ckpt_off), _ptr(ckpt_pos), n_ckpt,
                                     _ptr(ckpt_page), _ptr(o), H, d, int(n_segments), _ptr(workspace), ws_bytes,
                                     _ptr(dev_status), _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_prefill_paged")
    return o


def decode_paged_workspace_size(n_pages) -> int:
    return int(library().kda_decode_paged_workspace_size(int(n_pages)))


def decode_paged(q, k, v, g, beta, state_pool, s_in_page, s_out_page=None, n_commit=None, o=None, workspace=None,
                 dev_status=None, stream=None):
    """:func:`decode` with the states in a page pool (``kda_decode_paged``).

    s_in_page ``[B * H]`` int32 (entry ``b * H + h``; -1 = a zero state); s_out_page the
    same, or None to update in place.  A destination other than the source receives the
    state after ``n_commit[b]`` tokens (the entry state when that is 0).  Returns ``o``.
    """
    B, n_tok, H, d = q.shape
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape)
    _need(beta, "beta", torch.float32, (B, n_tok, H))
    n_pages = _pool(state_pool, d)
    _need(s_in_page, "s_in_page", torch.int32, (B * H,))
    _table(s_out_page, "s_out_page", B * H)
    if n_commit is not None:
        _need(n_commit, "n_commit", torch.int32, (B,))
    if o is None:
        o = torch.empty((B, n_tok, H, d), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32, (B, n_tok, H, d))
    if workspace is None:
        workspace = torch.empty(decode_paged_workspace_size(n_pages), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    st = library().kda_decode_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool), n_pages,
                                    _ptr(s_in_page), _ptr(s_out_page), _ptr(n_commit), _ptr(o), B, n_tok, H, d,
                                    _ptr(workspace), ws_bytes, _ptr(dev_status), _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_decode_paged")
    return o


def _host(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def prefill_host_blocks(cu_seqlens, block_tokens=0):
    """The block borders of :func:`prefill_host` for a host ``cu_seqlens`` (a list)."""
    _host(cu_seqlens, "cu_seqlens", torch.int32)
    n_seq = cu_seqlens.shape[0] - 1
    T = int(cu_seqlens[-1]) if n_seq >= 0 else 0
    out = torch.zeros(66, dtype=torch.int64)
    n = library().kda_prefill_host_blocks(_ptr(cu_seqlens), n_seq, T, int(block_tokens), _ptr(out), 66)
    if n < 0:
        raise ValueError("bad packing, block size, or more than 64 blocks")
    return out[:n + 1].tolist() if n > 0 else []


def prefill_host_workspace_size(n_seq, H, total_tokens, block_tokens=0, d=HEAD_DIM) -> int:
    return int(library().kda_prefill_host_workspace_size(int(n_seq), int(H), int(d), int(total_tokens),
                                                         int(block_tokens)))


def prefill_host(q, k, v, g, beta, cu_seqlens, S_in=None, o=None, S_out=None, block_tokens=0, workspace=None,
                 dev_status=None, stream=None):
    """:func:`prefill` from host tensors (``kda_prefill_host``): uploads, computes and downloads
    in pipelined blocks.  q, k, v, g, beta, S_in, o, S_out are HOST tensors (pinned for
    overlap); cu_seqlens a host int32 tensor.  ``workspace`` is a device uint8 tensor (made
    here when absent).  Returns ``(o, S_out)``; they are complete once ``stream`` is
    synchronised."""
    T, H, d = q.shape
    _host(q, "q", torch.bfloat16)
    _host(k, "k", torch.bfloat16, q.shape)
    _host(v, "v", torch.bfloat16, q.shape)
    _host(g, "g", torch.float32, q.shape)
    _host(beta, "beta", torch.float32, (T, H))
    _host(cu_seqlens, "cu_seqlens", torch.int32)
    n_seq = cu_seqlens.shape[0] - 1
    if S_in is not None:
        _host(S_in, "S_in", torch.float32, (n_seq, H, d, d))
    if o is None:
        o = torch.empty((T, H, d), dtype=torch.bfloat16).pin_memory()
    _host(o, "o", torch.bfloat16, (T, H, d))
    if S_out is None:
        S_out = torch.empty((n_seq, H, d, d), dtype=torch.float32).pin_memory()
    _host(S_out, "S_out", torch.float32, (n_seq, H, d, d))
    dev = torch.device("cuda", torch.cuda.current_device()) if stream is None else stream.device
    if workspace is None:
        workspace = torch.empty(prefill_host_workspace_size(n_seq, H, T, block_tokens, d), dtype=torch.uint8,
                                device=dev)
    _need(workspace, "workspace", torch.uint8)
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    st = library().kda_prefill_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S_in), _ptr(cu_seqlens),
                                    n_seq, T, _ptr(o), _ptr(S_out), H, d, int(block_tokens), _ptr(workspace),
                                    workspace.numel(), _ptr(dev_status), _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_prefill_host")
    return o, S_out


def debug_stall_next_prefill(chunk):
    """Test hook (``kda_debug_stall_next_prefill``): the next prefill launch withholds one
    hand-off at ``chunk`` and gives up its waits after 4096 polls, so it reports
    KDA_ERR_TIMEOUT in ``dev_status`` without any fault."""
    library().kda_debug_stall_next_prefill(int(chunk))


NOALLOC_SCRATCH_BYTES = 32 << 20


def prefill_noalloc(q, k, v, g, beta, cu_seqlens, S_in=None, ckpt_off=None, ckpt_pos=None, o=None, S_out=None,
                    ckpts=None, n_segments=0, dev_status=None, stream=None):
    """:func:`prefill` for callers that cannot allocate device memory (``kda_prefill_noalloc``).

    The library takes its scratch from a fixed 32 MiB array of its own instead of a
    caller-provided workspace; larger problems raise ``KdaError`` (KDA_ERR_WORKSPACE).
    Output tensors are created here only when not given; pass them in to allocate nothing.
    Calls share the array: do not let two of them overlap on the GPU.
    """
    T, H, d = q.shape
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape)
    _need(beta, "beta", torch.float32, (T, H))
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    n_seq = cu_seqlens.shape[0] - 1
    if S_in is not None:
        _need(S_in, "S_in", torch.float32, (n_seq, H, d, d))
    n_ckpt = 0
    if ckpt_off is not None:
        _need(ckpt_off, "ckpt_off", torch.int32, (n_seq + 1,))
        _need(ckpt_pos, "ckpt_pos", torch.int32)
        n_ckpt = ckpt_pos.shape[0]
        if ckpts is None:
            ckpts = torch.empty((n_ckpt, H, d, d), dtype=torch.float32, device=q.device)
        _need(ckpts, "ckpts", torch.float32, (n_ckpt, H, d, d))
    if o is None:
        o = torch.empty((T, H, d), dtype=torch.bfloat16, device=q.device)
    _need(o, "o", torch.bfloat16, (T, H, d))
    if S_out is None:
        S_out = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=q.device)
    _need(S_out, "S_out", torch.float32, (n_seq, H, d, d))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    st = library().kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S_in),
                                       _ptr(cu_seqlens), n_seq, T, _ptr(ckpt_off), _ptr(ckpt_pos), n_ckpt, _ptr(o),
                                       _ptr(S_out), _ptr(ckpts), H, d, int(n_segments), _ptr(dev_status),
                                       _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_prefill_noalloc")
    return o, S_out, ckpts


def prefill_pairs(q, k, v, g, beta, cu_seqlens, M=None, S_tilde=None, dev_status=None, stream=None):
    """Per (sequence, head), the pair (M, S~) of the sequence's rows (``kda_prefill_pairs``):
    the cumulative transition and the state from a zero entry state.  Inputs as
    :func:`prefill`.  Returns ``(M, S_tilde)``, each ``[N, H, 128, 128]`` fp32."""
    T, H, d = q.shape
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape)
    _need(beta, "beta", torch.float32, (T, H))
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    n_seq = cu_seqlens.shape[0] - 1
    if M is None:
        M = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=q.device)
    if S_tilde is None:
        S_tilde = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=q.device)
    _need(M, "M", torch.float32, (n_seq, H, d, d))
    _need(S_tilde, "S_tilde", torch.float32, (n_seq, H, d, d))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32)
    st = library().kda_prefill_pairs(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), n_seq, T,
                                     _ptr(M), _ptr(S_tilde), H, d, _ptr(dev_status), _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_prefill_pairs")
    return M, S_tilde


def combine_pairs(M, S_tilde, S_in=None, entry=None, stream=None):
    """Entry states after the ranges whose pairs are given (``kda_combine_pairs``): M and
    S_tilde ``[R, N, H, 128, 128]`` fp32 (R >= 0), S_in ``[N, H, 128, 128]`` or None (zeros).
    Returns ``entry`` ``[N, H, 128, 128]``: E = S_in, then E = S~_r + M_r E for r = 0 .. R-1."""
    _need(M, "M", torch.float32)
    if M.dim() != 5:
        raise ValueError(f"M must have shape [R, N, H, d, d], got {tuple(M.shape)}")
    R, n_seq, H, d, _ = M.shape
    _need(S_tilde, "S_tilde", torch.float32, M.shape)
    if S_in is not None:
        _need(S_in, "S_in", torch.float32, (n_seq, H, d, d))
    if entry is None:
        entry = torch.empty((n_seq, H, d, d), dtype=torch.float32, device=M.device)
    _need(entry, "entry", torch.float32, (n_seq, H, d, d))
    st = library().kda_combine_pairs(_ptr(M) if R else None, _ptr(S_tilde) if R else None, R, _ptr(S_in),
                                     _ptr(entry), n_seq, H, d, _stream_handle(stream))
    if st != 0:
        raise KdaError(st, "kda_combine_pairs")
    return entry
