"""Fused output stage (kda_prefill_gated) against the fp64 oracle, through the C ABI.

"Kimi K3.1 Pro 架构完全拆解" section 3.3: y = W_o [Sigmoid(W_g x) (.) RMSNorm(o~)]; the
library computes the bracket from supplied gate logits.  Reference: the oracle's fp64
recurrence output o~ passed through ``oracle.epilogue.gated_rmsnorm``.

The pages fix no tolerance for y.  The bar (``kda_gpu_util.y_bound``, derived there and
itself tested on the CPU in ``test_output_bar.py``) is the o bar carried through the output
stage exactly, plus y's own bf16 rounding: it says nothing about how an implementation
forms the stage.  State outputs are unchanged by the output stage (bit for bit against
kda_prefill); varlen boundaries bit-exact (packed == standalone, no write outside a
sequence's rows)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device, y_bound

pytestmark = pytest.mark.gpu
EPS = 1e-5


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
    """The bar of the module docstring; returns (e_o, worst |y - y_ref| / bound, e_s), and
    prints max|y - y_ref| / max|y_ref| as a diagnostic."""
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
            rows.append((host(y[a:b:o_stride, h]), r["o"], host(gate[a:b:o_stride, h])))
    e_o = rel_max(np.concatenate(og), np.concatenate(orf))
    assert e_o <= O_TOL, f"o error {e_o:.3e}"
    omax = np.abs(np.concatenate(orf)).max()
    worst, num, den = 0.0, 0.0, 0.0
    for yk, oref, gl in rows:
        bound, yr = y_bound(oref, gl, w, eps, omax)
        worst = max(worst, float((np.abs(yk - yr) / bound).max()))
        num, den = max(num, float(np.abs(yk - yr).max())), max(den, float(np.abs(yr).max()))
    assert worst <= 1.0, f"y off the oracle by {worst:.2f} x its bound"
    e_s = rel_fro(np.stack(sg), np.stack(sr))
    assert e_s <= S_TOL, f"state error {e_s:.3e}"
    print(f"e_o {e_o:.3e}  y/bound {worst:.3f}  max|y-y_ref|/max|y_ref| {num / den:.3e}  e_s {e_s:.3e}")
    return e_o, worst, e_s


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
