"""Seeded synthetic inputs shaped like the KDA workloads.

This module holds none of the method's arithmetic: it only draws random tensors in the
layouts the library and the oracle both take, so that the same values reach both.

Layouts (token-major, head-contiguous):
    q, k, v : [T_tot, H, d]   bfloat16   (decode: [B, n_tok, H, d])
    g       : [T_tot, H, d]   float32    natural-log per-channel decay
    beta    : [T_tot, H]      float32
    S0      : [N, H, d, d]    float32    (row = d_k channel, column = d_v) or None

Distributions (per element, in this draw order: lengths, q, k, v, beta-logits,
g-logits, S0):
    q, k  ~ N(0, 1), L2-normalised over d per (token, head) in float32, then bf16 (RNE)
    v     ~ N(0, 1) -> bf16
    beta  = sigmoid(N(0, 1))
    g     = -5 * sigmoid(N(0, 1) - 4)          ("sigmoid" decay: typical g ~ -0.09)
          or uniform on [-5, 0)                ("uniform" decay: the stress case)
    S0    ~ N(0, 0.02^2) when requested
The -5 floor is the bounded log-decay of "Kimi K3.1 Pro 架构完全拆解" section 3.2
(g_min = -5, alpha >= e^-5 ~ 6.7e-3).

Packed (varlen) inputs draw each sequence from its own generator seeded
``1000 * seed + i``, so one sequence can be regenerated alone.

Output stage ("Kimi K3.1 Pro 架构完全拆解" section 3.3): gate logits [T_tot, H, d] bf16
~ N(0, 1) (the projection W_g x of a unit-scale input) and a RMSNorm weight [d] float32
~ 1 + 0.1 N(0, 1), from their own generator (``make_output_stage``).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

G_MIN = -5.0


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    S0: torch.Tensor | None
    cu_seqlens: torch.Tensor            # int32 [N+1] (host)
    ckpt_off: torch.Tensor | None = None  # int32 [N+1] (host)
    ckpt_pos: torch.Tensor | None = None  # int32 [n_ckpt] (host)
    meta: dict = field(default_factory=dict)

    @property
    def n_seq(self) -> int:
        return int(self.cu_seqlens.numel()) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])


@dataclass
class DecodeInputs:
    q: torch.Tensor       # [B, n_tok, H, d] bf16
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor       # [B, n_tok, H, d] f32
    beta: torch.Tensor    # [B, n_tok, H] f32
    S0: torch.Tensor      # [B, H, d, d] f32
    n_commit: torch.Tensor | None  # int32 [B] (host) or None (= n_tok)
    meta: dict = field(default_factory=dict)


def _gen(device, seed):
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return gen


def _unit_rows(x):
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def _draw_tokens(shape_tok, H, d, gen, device, decay):
    """q, k, v, beta, g for ``shape_tok`` leading token dims, in the fixed draw order."""
    shp = tuple(shape_tok) + (H, d)
    q = _unit_rows(torch.randn(shp, generator=gen, device=device)).to(torch.bfloat16)
    k = _unit_rows(torch.randn(shp, generator=gen, device=device)).to(torch.bfloat16)
    v = torch.randn(shp, generator=gen, device=device).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn(tuple(shape_tok) + (H,), generator=gen, device=device))
    if decay == "sigmoid":
        g = G_MIN * torch.sigmoid(torch.randn(shp, generator=gen, device=device) - 4.0)
    elif decay == "uniform":
        g = G_MIN * (1.0 - torch.rand(shp, generator=gen, device=device))
    else:
        raise ValueError(f"unknown decay distribution {decay!r}")
    return q, k, v, beta, g


def checkpoint_positions(lengths, every):
    """Every multiple of ``every`` in (0, len] per sequence, as CSR (off, pos)."""
    off = [0]
    pos = []
    for n in lengths:
        pos.extend(range(every, int(n) + 1, every))
        off.append(len(pos))
    return torch.tensor(off, dtype=torch.int32), torch.tensor(pos, dtype=torch.int32)


def make_prefill(lengths, H, d=128, seed=0, device="cpu", decay="sigmoid", s0_std=None,
                 ckpt_every=None):
    """Packed prefill inputs for sequences of the given lengths.

    A single sequence is drawn from ``seed`` directly; several sequences are drawn one by
    one from sub-seeds ``1000 * seed + i``.
    """
    lengths = [int(n) for n in lengths]
    parts = []
    for i, n in enumerate(lengths):
        gen = _gen(device, seed if len(lengths) == 1 else 1000 * seed + i)
        q, k, v, beta, g = _draw_tokens((n,), H, d, gen, device, decay)
        S0 = None
        if s0_std is not None:
            S0 = torch.randn((1, H, d, d), generator=gen, device=device) * s0_std
        parts.append((q, k, v, beta, g, S0))
    cat = lambda j: torch.cat([p[j] for p in parts], 0) if parts else None
    q, k, v, beta, g = (cat(j) for j in range(5))
    S0 = torch.cat([p[5] for p in parts], 0) if s0_std is not None else None
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    off = pos = None
    if ckpt_every:
        off, pos = checkpoint_positions(lengths, ckpt_every)
    return PrefillInputs(q, k, v, g, beta, S0, cu, off, pos,
                         meta=dict(lengths=lengths, H=H, d=d, seed=seed, decay=decay,
                                   s0_std=s0_std, ckpt_every=ckpt_every, device=str(device)))


def make_output_stage(T, H, d=128, seed=0, device="cpu"):
    """Gate logits ``[T, H, d]`` bf16 and RMSNorm weight ``[d]`` float32 for the fused output
    stage, from a generator seeded ``7919 + seed`` (independent of the token draws)."""
    gen = _gen(device, 7919 + seed)
    gate = torch.randn((T, H, d), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    weight = 1.0 + 0.1 * torch.randn((d,), generator=gen, device=device, dtype=torch.float32)
    return gate, weight


@dataclass
class FrontEndInputs:
    qp: torch.Tensor          # [B, n_tok, H, d] bf16 projected inputs
    kp: torch.Tensor
    vp: torch.Tensor
    conv_w: torch.Tensor      # [3, H, d, W] fp32
    conv_cache: torch.Tensor  # [B, H, 3, W - 1, d] fp32 (bf16-representable past inputs)
    z: torch.Tensor           # [B, n_tok, H, d] fp32 decay-gate pre-activations
    a_log: torch.Tensor       # [H] fp32
    b: torch.Tensor           # [B, n_tok, H] fp32 beta logits
    S0: torch.Tensor          # [B, H, d, d] fp32
    n_commit: torch.Tensor | None
    gate: torch.Tensor        # [B, n_tok, H, d] bf16 output-gate logits
    norm_weight: torch.Tensor  # [d] fp32


def make_decode_frontend(B, n_tok, H, W=4, d=128, seed=0, device="cpu", commit="all", s0_std=0.02):
    """Inputs of a fused decode / verify step from projected inputs.  Draw order: qp, kp, vp,
    conv filters, cache, z, a_log, b, S0, gate, norm weight; then n_commit (as make_decode).
    qp, kp, vp ~ N(0, 1) -> bf16; filters ~ N(0, 0.5^2); the cache holds bf16-rounded N(0, 1)
    past inputs; z ~ N(-4, 1) and a_log ~ N(0, 0.1^2), so that g = -5 Sigmoid(e^a z) is
    typically about -0.09 like the other decode inputs; b ~ N(0, 1); S0 ~ N(0, s0_std^2)."""
    gen = _gen(device, 31337 + seed)
    rn = lambda *shape: torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    qp, kp, vp = (rn(B, n_tok, H, d).to(torch.bfloat16) for _ in range(3))
    conv_w = rn(3, H, d, W) * 0.5
    conv_cache = rn(B, H, 3, W - 1, d).to(torch.bfloat16).float()
    z = rn(B, n_tok, H, d) - 4.0
    a_log = rn(H) * 0.1
    b = rn(B, n_tok, H)
    S0 = rn(B, H, d, d) * s0_std
    gate = rn(B, n_tok, H, d).to(torch.bfloat16)
    norm_weight = 1.0 + 0.1 * rn(d)
    n_commit = None
    if commit == "random":
        n_commit = torch.randint(0, n_tok + 1, (B,), generator=_gen("cpu", 7919 * seed + 3),
                                 dtype=torch.int64).to(torch.int32)
    elif commit != "all":
        raise ValueError(commit)
    return FrontEndInputs(qp, kp, vp, conv_w, conv_cache, z, a_log, b, S0, n_commit, gate, norm_weight)


def make_page_tables(counts, n_pages, seed=0):
    """Distinct pages for several int32 page tables: ``counts`` entries each, drawn without
    replacement from a seeded permutation of ``range(n_pages)`` (scattered over the pool)."""
    total = sum(int(c) for c in counts)
    if total > n_pages:
        raise ValueError(f"{total} pages asked of a pool of {n_pages}")
    perm = torch.randperm(n_pages, generator=_gen("cpu", 104729 + seed)).to(torch.int32)
    out, at = [], 0
    for c in counts:
        out.append(perm[at:at + int(c)].clone())
        at += int(c)
    return out


def varlen_lengths(n_seq, lo, hi, seed):
    """Sequence lengths uniform on {lo, ..., hi}, drawn first from ``seed``."""
    gen = _gen("cpu", seed)
    return torch.randint(lo, hi + 1, (n_seq,), generator=gen).tolist()


def make_decode(B, n_tok, H, d=128, seed=0, device="cpu", s0_std=0.02, commit="all"):
    """Decode / verify inputs: ``commit`` is "all" (n_commit = n_tok) or "random"
    (n_commit uniform on {0, ..., n_tok}, drawn after S0)."""
    gen = _gen(device, seed)
    q, k, v, beta, g = _draw_tokens((B, n_tok), H, d, gen, device, "sigmoid")
    S0 = torch.randn((B, H, d, d), generator=gen, device=device) * s0_std
    n_commit = None
    if commit == "random":
        n_commit = torch.randint(0, n_tok + 1, (B,), generator=_gen("cpu", 7919 * seed + 1),
                                 dtype=torch.int64).to(torch.int32)
    elif commit != "all":
        raise ValueError(commit)
    return DecodeInputs(q, k, v, g, beta, S0, n_commit,
                        meta=dict(B=B, n_tok=n_tok, H=H, d=d, seed=seed, commit=commit))


# The workloads, by name.  Sizes follow the pages' model width (96 heads of 128, up to
# 1M tokens; "Kimi K3.1 Pro 架构完全拆解" section 2.3).
WORKLOADS = {
    "tiny": dict(kind="prefill", lengths=[256], H=2, seed=0, decay="sigmoid", s0_std=None),
    "prefill_8k": dict(kind="prefill", lengths=[8192], H=96, seed=1, decay="sigmoid", s0_std=None),
    "prefill_1m": dict(kind="prefill", lengths=[1 << 20], H=8, seed=2, decay="sigmoid", s0_std=None),
    "decode": dict(kind="decode", B=256, n_tok=1, H=96, seed=3),
    "verify": dict(kind="decode", B=256, n_tok=4, H=96, seed=3, commit="random"),
    "varlen": dict(kind="prefill", n_seq=64, len_lo=512, len_hi=16384, H=96, seed=4,
                   decay="uniform", s0_std=0.02, ckpt_every=512),
}


def make_workload(name, device="cpu", **over):
    w = dict(WORKLOADS[name])
    w.update(over)
    if w["kind"] == "decode":
        return make_decode(w["B"], w["n_tok"], w["H"], seed=w["seed"], device=device,
                           commit=w.get("commit", "all"))
    lengths = w.get("lengths")
    if lengths is None:
        lengths = varlen_lengths(w["n_seq"], w["len_lo"], w["len_hi"], w["seed"])
    return make_prefill(lengths, w["H"], seed=w["seed"], device=device, decay=w["decay"],
                        s0_std=w.get("s0_std"), ckpt_every=w.get("ckpt_every"))
