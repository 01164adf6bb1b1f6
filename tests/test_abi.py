"""The C-ABI library: it loads, exports what include/kda.h declares, and rejects bad
arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

OK, INVALID, UNSUPPORTED, ALIGNMENT, WORKSPACE, CUDA = 0, 1, 2, 3, 4, 5
HAS_GPU = torch.cuda.is_available()


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kda.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"kda_prefill", "kda_decode", "kda_prefill_workspace_size", "kda_status_string"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", kda.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out.stdout, flags=re.M))
    for n in names:
        assert n in exported, f"{n} declared in kda.h but not exported"
        getattr(lib, n)


def test_library_does_not_link_the_oracle(lib):
    out = subprocess.run(["nm", "-D", kda.LIB_PATH], capture_output=True, text=True, check=True).stdout
    assert "kda_ref_" not in out
    pkg = os.path.join(ROOT, "kimi_delta_attention_prefill_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "kda_oracle" not in src, f


def test_status_strings(lib):
    assert kda.status_string(0) == "KDA_OK"
    assert kda.status_string(6) == "KDA_ERR_TIMEOUT"
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"
    assert kda.version() >= 100


P = lambda a: ctypes.c_void_p(a)


def _decode(lib, B=2, n_tok=1, H=3, d=128, q=0x1000, S=0x2000, beta=0x3000, n_commit=None, o=0x4000):
    return lib.kda_decode(P(q), P(0x5000), P(0x6000), P(0x7000), P(beta), P(S), n_commit, P(o), B, n_tok, H, d,
                          None, None)


def test_decode_host_validation(lib):
    assert _decode(lib, d=64) == UNSUPPORTED
    assert _decode(lib, n_tok=0) == UNSUPPORTED
    assert _decode(lib, n_tok=5) == UNSUPPORTED
    assert _decode(lib, B=-1) == INVALID
    assert _decode(lib, B=0) == OK and _decode(lib, H=0) == OK  # empty: no-op
    assert _decode(lib, q=0) == INVALID
    assert _decode(lib, S=0) == INVALID
    assert _decode(lib, q=0x1002) == ALIGNMENT
    assert _decode(lib, S=0x2008) == ALIGNMENT
    assert _decode(lib, beta=0x3002) == ALIGNMENT
    if not HAS_GPU:
        assert _decode(lib) in (CUDA, UNSUPPORTED)


def _prefill(lib, n_seq=1, T=64, H=2, d=128, cu=0x9000, q=0x1000, ckpt_off=None, ckpt_pos=None, n_ckpt=0,
             ckpts=None, n_segments=0, ws=None, ws_bytes=0):
    return lib.kda_prefill(P(q), P(0x1100), P(0x1200), P(0x1300), P(0x1400), None, P(cu), n_seq, T,
                           ckpt_off, ckpt_pos, n_ckpt, P(0x1500), P(0x1600), ckpts, H, d, n_segments, ws,
                           ws_bytes, None, None)


def test_prefill_host_validation(lib):
    assert _prefill(lib, d=96) == UNSUPPORTED
    assert _prefill(lib, n_seq=-1) == INVALID
    assert _prefill(lib, T=-5) == INVALID
    assert _prefill(lib, n_segments=-1) == INVALID
    assert _prefill(lib, n_seq=0) == OK and _prefill(lib, H=0) == OK
    assert _prefill(lib, cu=0) == INVALID
    assert _prefill(lib, q=0) == INVALID
    assert _prefill(lib, n_ckpt=3) == INVALID                      # positions without offsets
    assert _prefill(lib, ckpt_off=P(0xA000), n_ckpt=3) == INVALID  # offsets without positions / slots
    assert _prefill(lib, q=0x1008) == ALIGNMENT
    assert _prefill(lib, cu=0x9002) == ALIGNMENT
    if not HAS_GPU:
        assert _prefill(lib) in (CUDA, UNSUPPORTED)


def _prefill_gated(lib, gate=0x1700, nw=None, eps=1e-5, q=0x1000, d=128, T=64):
    return lib.kda_prefill_gated(P(q), P(0x1100), P(0x1200), P(0x1300), P(0x1400), P(gate) if gate else None,
                                 P(nw) if nw else None, eps, None, P(0x9000), 1, T, None, None, 0, P(0x1500),
                                 P(0x1600), None, 2, d, 0, None, 0, None, None)


def test_prefill_gated_host_validation(lib):
    """The fused output stage ("Kimi K3.1 Pro 架构完全拆解" 3.3): bad eps, a missing or
    misaligned gate / weight are rejected before any CUDA call; the rest is kda_prefill's."""
    assert _prefill_gated(lib, eps=-1e-6) == INVALID
    assert _prefill_gated(lib, eps=float("nan")) == INVALID
    assert _prefill_gated(lib, eps=float("inf")) == INVALID
    assert _prefill_gated(lib, gate=0) == INVALID
    assert _prefill_gated(lib, gate=0x1708) == ALIGNMENT
    assert _prefill_gated(lib, nw=0x1804) == ALIGNMENT
    assert _prefill_gated(lib, d=64) == UNSUPPORTED
    assert _prefill_gated(lib, q=0) == INVALID
    if not HAS_GPU:
        assert _prefill_gated(lib) in (CUDA, UNSUPPORTED)
        assert _prefill_gated(lib, nw=0x1800, eps=0.0) in (CUDA, UNSUPPORTED)


def test_binding_rejects_cpu_tensors(lib):
    x = torch.zeros(4, 1, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.decode(x, x, x, x.float(), torch.zeros(4, 1, 2), torch.zeros(4, 2, 128, 128))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(kda.KdaLibraryError):
        kda.library()


def _split_bytes(n_seq, H, extra):
    """The split workspace for `extra` extra segments (layout in kda_internal.h: counts,
    two item tables, per-sequence info, then [slots][H][3][128][128] fp32)."""
    up = lambda x: (x + 255) // 256 * 256
    max1, max3 = n_seq + 2 * extra, extra
    n_slots = min(2 * extra, n_seq + extra)
    off3 = up(256 + 16 * max1)
    offs = up(off3 + 16 * max3)
    offsl = up(offs + 8 * n_seq)
    return offsl + n_slots * H * 3 * 128 * 128 * 4


def test_planner_wave_model(lib):
    """The automatic segment count minimises (w1 + w3) / (n - 1 + w1), w1 = ceil(H(2n-3)/S)
    pass-1 waves (the first segment, w1 times as long as the others, runs through all of
    them) and w3 = ceil(H(n-1)/S) pass-3 waves, with S = 152 (the library's assumption
    without a GPU); worked by hand:
    H = 8, 2^20 tokens: n = 20 (pass 1: 296 items = 2 waves, pass 3: 152 = 1 wave, 3/21);
    n = 19 would give 3/20 and n = 21 (3 + 2)/23.  H = 16: n = 10 (272 and 144 items, 3/11;
    9 gives 3/10).  One head, 9000 tokens: at most 2 segments by length, and 2 segments cost
    2/2 = 1, a tie with no split, which the planner keeps."""
    assert kda.prefill_workspace_size(1, 8, 1 << 20) == _split_bytes(1, 8, 19)
    assert kda.prefill_workspace_size(1, 16, 1 << 20) == _split_bytes(1, 16, 9)
    assert kda.prefill_workspace_size(1, 1, 9000) == 0
    # a forced count is taken as given (bounded by the chunks)
    assert kda.prefill_workspace_size(1, 8, 1 << 20, n_segments=19) == _split_bytes(1, 8, 18)


def test_workspace_sizes(lib):
    # without a GPU the library assumes 152 SMs for the planner's bound
    assert kda.prefill_workspace_size(1, 96, 8192) == 0
    assert kda.prefill_workspace_size(1, 8, 1 << 20) > 0
    assert kda.prefill_workspace_size(4, 2, 10000, n_segments=1) == 0
    assert kda.prefill_workspace_size(4, 2, 10000, n_segments=3) > 0
    assert kda.prefill_workspace_size(4, 2, 10000, n_segments=-1) == 0


def _prefill_paged(lib, pool=0x20000, n_pages=16, s_in=0xB000, s_out=0xB100, ckpt_off=None, ckpt_pos=None,
                   n_ckpt=0, ckpt_page=None, ws=0x40000, ws_bytes=1 << 20, gate=None, eps=1e-5, n_seq=1, H=2):
    return lib.kda_prefill_paged(P(0x1000), P(0x1100), P(0x1200), P(0x1300), P(0x1400), P(gate) if gate else None,
                                 None, eps, P(pool) if pool else None, n_pages, P(s_in) if s_in else None,
                                 P(s_out) if s_out else None, P(0x9000), n_seq, 64, ckpt_off, ckpt_pos, n_ckpt,
                                 P(ckpt_page) if ckpt_page else None, P(0x1500), H, 128, 0,
                                 P(ws) if ws else None, ws_bytes, None, None)


def test_prefill_paged_host_validation(lib):
    """Paged states ("部署 Kimi K3 ..." 3): a pool, int32 page tables, a workspace that always
    holds the page check; bad pools, tables and workspaces are rejected on the host."""
    assert _prefill_paged(lib, n_pages=-1) == INVALID
    assert _prefill_paged(lib, n_pages=1 << 31) == INVALID
    assert _prefill_paged(lib, pool=0) == INVALID
    assert _prefill_paged(lib, pool=0x20008) == ALIGNMENT
    assert _prefill_paged(lib, s_in=0xB002) == ALIGNMENT
    assert _prefill_paged(lib, ws=0x40010) == ALIGNMENT
    assert _prefill_paged(lib, ws=0, ws_bytes=0) == WORKSPACE
    assert _prefill_paged(lib, ws_bytes=100) == WORKSPACE
    assert _prefill_paged(lib, ckpt_off=P(0xA000), ckpt_pos=P(0xA100), n_ckpt=2) == INVALID  # no checkpoint pages
    assert _prefill_paged(lib, gate=0x1700, eps=-1.0) == INVALID
    assert _prefill_paged(lib, gate=0x1702) == ALIGNMENT
    assert _prefill_paged(lib, n_seq=0) == OK
    if not HAS_GPU:
        assert _prefill_paged(lib) in (CUDA, UNSUPPORTED)
        assert _prefill_paged(lib, s_in=0, s_out=0) in (CUDA, UNSUPPORTED)


def _decode_paged(lib, pool=0x20000, n_pages=16, s_in=0xB000, s_out=None, ws=0x40000, ws_bytes=1 << 20, n_tok=1,
                  B=2, H=2):
    return lib.kda_decode_paged(P(0x1000), P(0x1100), P(0x1200), P(0x1300), P(0x1400), P(pool) if pool else None,
                                n_pages, P(s_in) if s_in else None, P(s_out) if s_out else None, None, P(0x1500),
                                B, n_tok, H, 128, P(ws) if ws else None, ws_bytes, None, None)


def test_decode_paged_host_validation(lib):
    assert _decode_paged(lib, n_tok=5) == UNSUPPORTED
    assert _decode_paged(lib, n_pages=-3) == INVALID
    assert _decode_paged(lib, pool=0) == INVALID
    assert _decode_paged(lib, s_in=0) == INVALID
    assert _decode_paged(lib, s_out=0xB102) == ALIGNMENT
    assert _decode_paged(lib, ws=0) == WORKSPACE
    assert _decode_paged(lib, ws_bytes=256) == WORKSPACE  # 16 pages need 256 + 64 bytes
    assert _decode_paged(lib, B=0) == OK
    if not HAS_GPU:
        assert _decode_paged(lib) in (CUDA, UNSUPPORTED)


def test_paged_workspace_sizes(lib):
    assert kda.decode_paged_workspace_size(0) == 256
    assert kda.decode_paged_workspace_size(1000) == 256 + 4000
    assert kda.prefill_paged_workspace_size(1, 96, 8192, n_pages=10) == 256 + 40  # no split at 96 heads
    split = kda.prefill_workspace_size(4, 2, 10000, n_segments=3)
    assert kda.prefill_paged_workspace_size(4, 2, 10000, n_pages=7, n_segments=3) == (split + 255) // 256 * 256 + 284


def _decode_fused(lib, W=4, act=0, g_min=-5.0, gate=None, eps=1e-5, cache=0x7000, n_tok=2, qp=0x1000, S=0x2000,
                  B=2, H=2):
    return lib.kda_decode_fused(P(qp) if qp else None, P(0x1100), P(0x1200), P(0x3000), P(cache) if cache else None,
                                W, act, P(0x4000), P(0x5000), g_min, P(0x6000), P(gate) if gate else None, None, eps,
                                P(S) if S else None, None, P(0x8000), B, n_tok, H, 128, None, None)


def test_decode_fused_host_validation(lib):
    """The fused decode front end ("Kimi K3.1 Pro 架构完全拆解" 3.4): widths, activation,
    decay bound, epsilon and buffers are checked before any CUDA call."""
    assert _decode_fused(lib, W=0) == UNSUPPORTED
    assert _decode_fused(lib, W=5) == UNSUPPORTED
    assert _decode_fused(lib, n_tok=5) == UNSUPPORTED
    assert _decode_fused(lib, act=2) == INVALID
    assert _decode_fused(lib, g_min=0.0) == INVALID
    assert _decode_fused(lib, g_min=float("-inf")) == INVALID
    assert _decode_fused(lib, gate=0x9000, eps=-1.0) == INVALID
    assert _decode_fused(lib, cache=0) == INVALID       # W > 1 needs the cache
    assert _decode_fused(lib, qp=0) == INVALID
    assert _decode_fused(lib, S=0x2008) == ALIGNMENT
    assert _decode_fused(lib, qp=0x1001) == ALIGNMENT
    assert _decode_fused(lib, B=0) == OK
    if not HAS_GPU:
        assert _decode_fused(lib) in (CUDA, UNSUPPORTED)
        assert _decode_fused(lib, W=1, cache=0) in (CUDA, UNSUPPORTED)


def test_prefill_from_host_buffers_validation(lib):
    """kda_prefill_host reads the offsets on the host to plan its blocks: a bad packing or
    block size is refused before any CUDA call."""
    import numpy as np
    cu = np.array([0, 64, 100], dtype=np.int32)
    bad = np.array([0, 70, 60], dtype=np.int32)
    f = lambda c, T=100, blk=0, ws=0x40000, wsb=1 << 30: lib.kda_prefill_host(
        P(0x1000), P(0x1100), P(0x1200), P(0x1300), P(0x1400), None, c.ctypes.data, 2, T, P(0x1500), P(0x1600), 2,
        128, blk, P(ws) if ws else None, wsb, None, None)
    assert f(bad) == INVALID
    assert f(cu, T=99) == INVALID          # cu[n] != total_tokens
    assert f(cu, blk=100) == INVALID       # not a multiple of 64
    assert f(cu, ws=0x40010) == ALIGNMENT
    if not HAS_GPU:
        assert f(cu) in (CUDA, UNSUPPORTED, WORKSPACE)
