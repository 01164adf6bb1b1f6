"""Fused output stage (kda_prefill_gated) against the fp64 oracle, through the C ABI.

"Kimi K3.1 Pro 架构完全拆解" section 3.3: y = W_o [Sigmoid(W_g x) (.) RMSNorm(o~)]; the
library computes the bracket from supplied gate logits.  Reference: the oracle's fp64
recurrence output o~ passed through ``oracle.epilogue.gated_rmsnorm`` (E below).

The pages fix no tolerance for y; the bar is derived from the arithmetic:
  * the factor f = w sigmoid(a) is formed in half precision (fp16 keeps 11 significant
    bits: u16 = 2^-11): the exponent x = |a| log2(e) is rounded to fp16 (relative error
    ln2 ulp16(x) / 2 in 2^-x), raised by ex2.approx.f16x2 (EX2_H below), and the sum 1 + e,
    the Newton reciprocal (within one ulp), the numerator product, w and the product with w
    round six more times: eps_f(a) = ln2 ulp16(x) / 2 + EX2_H + 6 u16 (factor_err);
    below fp16's normal range the factor is off by at most 2^-24 absolutely;
  * epilogue arithmetic: y against E applied to the plain kernel's own bf16 o.  o is o~
    rounded to nearest (bf16 keeps 8 significant bits: relative error u = 2^-8 per element),
    which moves each normalised element by at most a factor (1 + u) / (1 - u) = 1 + 7.84e-3
    (the element and the row's root mean square each move by at most u); y itself is rounded
    once more (u), so |y - E(o)| <= (1.2e-2 + eps_f) |E(o)| (+ 1e-6 max|E(o)| for the fp32
    arithmetic and the factor's absolute floor);
  * end to end: with the recurrence's error |d o~|_max <= O_TOL max|o~| (the o bar), element
    c of a row with root mean square r moves by at most
    s_c |d o~|_max / r x (1 + |o~_c| / r) to first order (s_c = sigmoid x weight; the
    second term is the row norm's own change), so
    |y - y_ref| <= s_c O_TOL max|o~_ref| / r (1 + |o~_ref,c| / r) + (4e-3 + eps_f) |y_ref| + 1e-6.
    Rows whose norm is far below the tensor's maximum get a correspondingly wide bound:
    normalising a row divides its absolute error by its own norm.
State outputs are unchanged by the output stage (bit for bit against kda_prefill); varlen
boundaries bit-exact (packed == standalone, no write outside a sequence's rows)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device
from oracle.epilogue import gated_rmsnorm

pytestmark = pytest.mark.gpu
EPS = 1e-5
# relative error bound of ex2.approx.f16x2 on x <= 0 with normal fp16 results: every such
# input swept once on a GB300 gave at most 2^-10.08 (at x = -0.990); 2^-9.9 is taken
EX2_H = 2.0 ** -9.9


def factor_err(gl):
    """eps_f of the module docstring, per gate logit."""
    x = np.abs(gl.astype(np.float64)) * np.log2(np.e)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(x, 2.0 ** -14))) - 10)
    return np.log(2.0) * ulp / 2 + EX2_H + 6 * 2.0 ** -11


def run(inp, gate, weight, eps=EPS, n_segments=0, o_pad=0, gated=True):
    d = to_device(inp)
    T, H, _ = inp.q.shape
    buf = torch.full((T + 2 * o_pad, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = buf[o_pad:o_pad + T]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(gate=gate.cuda(), norm_weight=None if weight is None else weight.cuda(), eps=eps) if gated else {}
    y, S, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S_in=d["S0"],
                           ckpt_off=d["ckpt_off"], ckpt_pos=d["ckpt_pos"], o=y, n_segments=n_segments,
                           dev_status=st, **kw)
    torch.cuda.synchronize()
    return y, S, ck, int(st.item()), buf


def check(inp, gate, weight, y, S, units=None, o_stride=1, eps=EPS):
    """The bar of the module docstring; returns (e_o, worst end-to-end error / its bound,
    worst epilogue error / its bound, e_s)."""
    n_seq, H = inp.n_seq, inp.q.shape[1]
    units = units or [(s, h) for s in range(n_seq) for h in range(H)]
    o_plain, S_plain, _, st, _ = run(inp, gate, weight, eps=eps, gated=False)
    assert st == 0
    ref = oracle_units(inp, units, o_stride=o_stride)
    cu = inp.cu_seqlens.tolist()
    w = np.ones(128) if weight is None else weight.double().numpy()
    og, orf, sg, sr, rows = [], [], [], [], []
    for (s, h), r in ref.items():
        a, b = cu[s], cu[s + 1]
        sg.append(host(S[s, h]))
        sr.append(r["S"])
        if b > a:
            og.append(host(o_plain[a:b:o_stride, h]))
            orf.append(r["o"])
            rows.append((host(y[a:b:o_stride, h]), host(o_plain[a:b:o_stride, h]), r["o"],
                         host(gate[a:b:o_stride, h])))
    e_o = rel_max(np.concatenate(og), np.concatenate(orf))
    assert e_o <= O_TOL, f"o error {e_o:.3e}"
    omax = np.abs(np.concatenate(orf)).max()
    worst_e2e = worst_epi = 0.0
    for yk, ok, oref, gl in rows:
        ye = gated_rmsnorm(ok, gl, w, eps)           # epilogue of the kernel's own o
        ef = factor_err(gl)
        bound_epi = (1.2e-2 + ef) * np.abs(ye) + 1e-6 * np.abs(ye).max()
        worst_epi = max(worst_epi, float((np.abs(yk - ye) / bound_epi).max()))
        yr = gated_rmsnorm(oref, gl, w, eps)
        sc = 1.0 / (1.0 + np.exp(-gl.astype(np.float64))) * np.abs(w)
        rms = np.sqrt(np.mean(oref ** 2, axis=1, keepdims=True) + eps)
        bound = sc * O_TOL * omax / rms * (1.0 + np.abs(oref) / rms) + (4e-3 + ef) * np.abs(yr) + 1e-6
        worst_e2e = max(worst_e2e, float((np.abs(yk - yr) / bound).max()))
    assert worst_epi <= 1.0, f"epilogue arithmetic off by {worst_epi:.2f} x its bound"
    assert worst_e2e <= 1.0, f"y off the oracle by {worst_e2e:.2f} x its bound"
    e_s = rel_fro(np.stack(sg), np.stack(sr))
    assert e_s <= S_TOL, f"state error {e_s:.3e}"
    print(f"e_o {e_o:.3e}  y/bound {worst_e2e:.3f}  epilogue/bound {worst_epi:.3f}  e_s {e_s:.3e}")
    return e_o, worst_e2e, worst_epi, e_s


def test_tiny_config_gated():
    inp = inputs.make_workload("tiny", device="cpu")
    gate, w = inputs.make_output_stage(inp.q.shape[0], inp.q.shape[1], seed=0)
    y, S, ck, st, _ = run(inp, gate, w)
    assert st == 0
    check(inp, gate, w, y, S)


@pytest.mark.parametrize("T", [1, 63, 65, 257])
def test_single_sequences_gated(T):
    inp = inputs.make_prefill([T], H=3, seed=500 + T, device="cpu", decay="uniform", s0_std=0.02)
    gate, w = inputs.make_output_stage(T, 3, seed=T)
    y, S, ck, st, _ = run(inp, gate, w)
    assert st == 0
    check(inp, gate, w, y, S)


def test_wide_gate_logits():
    """Logits of standard deviation 6: large exponents (rounded coarsely in fp16) and
    factors below fp16's normal range."""
    inp = inputs.make_prefill([200], H=2, seed=65, device="cpu", s0_std=0.02)
    gate, w = inputs.make_output_stage(200, 2, seed=65)
    gate = (gate.float() * 6.0).to(torch.bfloat16)
    y, S, ck, st, _ = run(inp, gate, w)
    assert st == 0
    check(inp, gate, w, y, S)


def test_unit_weight_and_eps_zero():
    """norm_weight = None means ones; eps = 0 is allowed (rows are never all-zero here)."""
    inp = inputs.make_prefill([130], H=2, seed=61, device="cpu", s0_std=0.02)
    gate, _ = inputs.make_output_stage(130, 2, seed=61)
    y, S, ck, st, _ = run(inp, gate, None, eps=0.0)
    assert st == 0
    check(inp, gate, None, y, S, eps=0.0)


def test_output_stage_leaves_the_state_alone():
    """The gated call's state outputs are the plain call's, bit for bit."""
    inp = inputs.make_prefill([5, 200, 64], H=2, seed=62, device="cpu", s0_std=0.02, ckpt_every=64)
    gate, w = inputs.make_output_stage(inp.q.shape[0], 2, seed=62)
    _, S1, ck1, st1, _ = run(inp, gate, w)
    _, S0, ck0, st0, _ = run(inp, gate, w, gated=False)
    assert st1 == 0 and st0 == 0
    assert torch.equal(S1, S0) and torch.equal(ck1, ck0)


def test_varlen_gated_boundaries():
    lens = [5, 64, 1, 130, 0, 77]
    inp = inputs.make_prefill(lens, H=2, seed=63, device="cpu", decay="uniform", s0_std=0.02)
    gate, w = inputs.make_output_stage(inp.q.shape[0], 2, seed=63)
    y, S, ck, st, buf = run(inp, gate, w, o_pad=64)
    assert st == 0
    check(inp, gate, w, y, S)
    assert torch.isnan(buf[:64].float()).all() and torch.isnan(buf[-64:].float()).all()
    cu = inp.cu_seqlens.tolist()
    for s in range(inp.n_seq):
        a, b = cu[s], cu[s + 1]
        one = inputs.PrefillInputs(inp.q[a:b], inp.k[a:b], inp.v[a:b], inp.g[a:b], inp.beta[a:b],
                                   inp.S0[s:s + 1], torch.tensor([0, b - a], dtype=torch.int32))
        y1, S1, _, st1, _ = run(one, gate[a:b], w)
        assert st1 == 0
        assert torch.equal(y1, y[a:b]) and torch.equal(S1[0], S[s])


@pytest.mark.parametrize("n_seg", [2, 5])
def test_split_path_gated(n_seg):
    """The sequence split (several segments) writes y in its first and last passes."""
    inp = inputs.make_prefill([1500], H=2, seed=64, device="cpu", s0_std=0.02)
    gate, w = inputs.make_output_stage(1500, 2, seed=64)
    y, S, ck, st, _ = run(inp, gate, w, n_segments=n_seg)
    assert st == 0
    check(inp, gate, w, y, S)


def test_prefill_8k_gated_sampled():
    """The benchmark's workload (1 x 8192, 96 heads) with the output stage: four heads
    against the oracle on every 8th row."""
    inp = inputs.make_workload("prefill_8k", device="cuda")
    gate, w = inputs.make_output_stage(8192, 96, seed=1, device="cuda")
    y, S, ck, st, _ = run(inp, gate, w)
    assert st == 0
    check(inp, gate.cpu(), w.cpu(), y, S, units=[(0, 0), (0, 31), (0, 64), (0, 95)], o_stride=8)
