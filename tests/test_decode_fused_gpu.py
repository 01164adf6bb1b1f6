"""Fused decode front end (kda_decode_fused) against the fp64 oracle, through the C ABI.

"Kimi K3.1 Pro 架构完全拆解" 3.4: the replay kernel of speculative decoding starts from the
cached projected inputs and does the short convolution, input normalisation, gating, the
recurrence and the output normalisation in one kernel; the steps follow "Kimi K3 ...
服務性能" section 7 and the K3.1 page 3.2 (``oracle.frontend.decode_step``).

Bar: the decode tolerance max|x - x_ref| / max|x_ref| <= 1e-4 on o and on the committed
state (fp32 in and out); the convolution cache is a copy of inputs, so it is bit-exact.
With the output stage, y = Sigmoid(gate) w o / r (r the row's root mean square): an error
of at most DECODE_TOL max|o_ref| in o moves element c by at most
s_c DECODE_TOL max|o_ref| / r (1 + |o_ref,c| / r) to first order (s_c = Sigmoid x weight),
plus the fp32 arithmetic of the stage (1e-5 |y| + 1e-7).
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import DECODE_TOL, host, rel_max
from oracle.frontend import decode_step

pytestmark = pytest.mark.gpu
DEVICE_CHECK = 7


def run(x, act="none", gated=False, units=None, dev_status=None):
    S = x.S0.cuda().clone()
    cache = x.conv_cache.cuda().clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if dev_status is None else dev_status
    kw = dict(gate=x.gate.cuda(), norm_weight=x.norm_weight.cuda()) if gated else {}
    o = kda.decode_fused(x.qp.cuda(), x.kp.cuda(), x.vp.cuda(), x.conv_w.cuda(), cache, x.z.cuda(), x.a_log.cuda(),
                         x.b.cuda(), S, n_commit=None if x.n_commit is None else x.n_commit.cuda(), conv_act=act,
                         dev_status=st, **kw)
    torch.cuda.synchronize()
    return o, S, cache, int(st.item())


def reference(x, act="none", gated=False, bsel=None):
    f = lambda t: host(t) if bsel is None else host(t[bsel])
    nc = None if x.n_commit is None else (x.n_commit.numpy() if bsel is None else x.n_commit.numpy()[bsel])
    return decode_step(f(x.qp), f(x.kp), f(x.vp), host(x.conv_w), f(x.conv_cache), f(x.z), host(x.a_log), f(x.b),
                       f(x.S0), n_commit=nc, act=act, gate=f(x.gate) if gated else None,
                       norm_weight=host(x.norm_weight) if gated else None, eps=1e-5)


def check(x, o, S, cache, ref, bsel=None):
    sel = (lambda t: host(t)) if bsel is None else (lambda t: host(t[bsel]))
    e_o = rel_max(sel(o), ref["o"])
    e_s = rel_max(sel(S), ref["S"])
    assert e_o <= DECODE_TOL, f"o error {e_o:.3e}"
    assert e_s <= DECODE_TOL, f"state error {e_s:.3e}"
    assert np.array_equal(sel(cache), ref["conv_cache"]), "convolution cache differs"
    return e_o, e_s


@pytest.mark.parametrize("W,act", [(1, "none"), (2, "silu"), (3, "none"), (4, "none"), (4, "silu")])
@pytest.mark.parametrize("n_tok,commit", [(1, "all"), (2, "random"), (3, "all"), (4, "random")])
def test_fused_step_against_oracle(W, act, n_tok, commit):
    x = inputs.make_decode_frontend(6, n_tok, 3, W=W, seed=10 * W + n_tok, commit=commit)
    o, S, cache, st = run(x, act)
    assert st == 0
    check(x, o, S, cache, reference(x, act))


@pytest.mark.parametrize("n_tok,commit", [(1, "all"), (4, "random")])
def test_fused_step_with_output_stage(n_tok, commit):
    x = inputs.make_decode_frontend(5, n_tok, 2, W=4, seed=40 + n_tok, commit=commit)
    o, S, cache, st = run(x, "silu", gated=True)
    assert st == 0
    ref_plain = reference(x, "silu")
    ref = reference(x, "silu", gated=True)
    y, yr, orf = host(o), ref["o"], ref_plain["o"]
    omax = np.abs(orf).max()
    rms = np.sqrt(np.mean(orf ** 2, axis=-1, keepdims=True) + 1e-5)
    sc = 1.0 / (1.0 + np.exp(-host(x.gate))) * host(x.norm_weight)
    bound = sc * DECODE_TOL * omax / rms * (1.0 + np.abs(orf) / rms) + 1e-5 * np.abs(yr) + 1e-7
    assert (np.abs(y - yr) / bound).max() <= 1.0
    assert rel_max(host(S), ref["S"]) <= DECODE_TOL
    assert np.array_equal(host(cache), ref["conv_cache"])


def test_two_steps_equal_one_step():
    """Replay identity: steps over tokens 0..1 then 2..3 (state and cache carried) give the
    outputs, state and cache of one step over tokens 0..3 (fp32 on both sides: tolerance)."""
    x = inputs.make_decode_frontend(4, 4, 2, W=4, seed=50, commit="all")
    o_all, S_all, c_all, st = run(x)
    assert st == 0
    part = lambda t, a, e: t[:, a:e].contiguous()
    x1 = inputs.FrontEndInputs(part(x.qp, 0, 2), part(x.kp, 0, 2), part(x.vp, 0, 2), x.conv_w, x.conv_cache,
                               part(x.z, 0, 2), x.a_log, part(x.b, 0, 2), x.S0, None, part(x.gate, 0, 2), x.norm_weight)
    o1, S1, c1, st1 = run(x1)
    x2 = inputs.FrontEndInputs(part(x.qp, 2, 4), part(x.kp, 2, 4), part(x.vp, 2, 4), x.conv_w, c1.cpu(),
                               part(x.z, 2, 4), x.a_log, part(x.b, 2, 4), S1.cpu(), None, part(x.gate, 2, 4),
                               x.norm_weight)
    o2, S2, c2, st2 = run(x2)
    assert st1 == 0 and st2 == 0
    assert torch.equal(c2, c_all)
    assert rel_max(host(torch.cat([o1, o2], 1)), host(o_all)) <= DECODE_TOL
    assert rel_max(host(S2), host(S_all)) <= DECODE_TOL


def test_bad_commit_leaves_state_and_cache():
    x = inputs.make_decode_frontend(3, 2, 2, W=3, seed=51, commit="all")
    x.n_commit = torch.tensor([2, 5, 1], dtype=torch.int32)  # 5 > n_tok
    o, S, cache, st = run(x)
    assert st == DEVICE_CHECK
    assert torch.equal(S[1].cpu(), x.S0[1]) and torch.equal(cache[1].cpu(), x.conv_cache[1])
    ref = reference(inputs.FrontEndInputs(*(getattr(x, f) for f in ("qp", "kp", "vp", "conv_w", "conv_cache", "z",
                                                                    "a_log", "b", "S0")),
                                          torch.tensor([2, 0, 1], dtype=torch.int32), x.gate, x.norm_weight))
    assert rel_max(host(o), ref["o"]) <= DECODE_TOL  # outputs are still produced for every sequence
    assert rel_max(host(S), ref["S"]) <= DECODE_TOL


def test_zero_projected_row_stays_zero():
    """A q / k whose convolution output is zero is left zero by the normalisation."""
    x = inputs.make_decode_frontend(2, 1, 2, W=1, seed=52)
    x.qp[0, 0, 1] = 0
    x.kp[1, 0, 0] = 0
    o, S, cache, st = run(x)
    assert st == 0
    check(x, o, S, cache, reference(x))


def test_verify_workload_sampled():
    """256 sequences x 96 heads, 4 tokens, random commits, W = 4 with SiLU, the output stage:
    the whole launch, checked on eight sequences (all heads) against the oracle."""
    x = inputs.make_decode_frontend(256, 4, 96, W=4, seed=53, commit="random", device="cpu")
    o, S, cache, st = run(x, "silu")
    assert st == 0
    bsel = np.array([0, 1, 37, 100, 128, 200, 254, 255])
    ref = reference(x, "silu", bsel=bsel)
    assert rel_max(host(o[bsel]), ref["o"]) <= DECODE_TOL
    assert rel_max(host(S[bsel]), ref["S"]) <= DECODE_TOL
    assert np.array_equal(host(cache[bsel]), ref["conv_cache"])


@pytest.mark.parametrize("z_val,b_val", [(30.0, 30.0), (-30.0, -30.0), (30.0, -30.0), (100.0, -100.0),
                                         (-100.0, 100.0)])
def test_saturated_gates(z_val, b_val):
    """z = +-30 puts the decay at g_min or 0 (alpha = e^-5 or 1), b = +-30 puts beta at 1 or
    0: the gates' saturated ends, against the oracle.  At +-100, e^-x overflows fp32 in the
    sigmoid's denominator (1 + e^100 = inf), which must give exactly 0, not a NaN."""
    x = inputs.make_decode_frontend(3, 4, 2, W=3, seed=54, commit="random")
    x.z.fill_(z_val)
    x.b.fill_(b_val)
    o, S, cache, st = run(x, "silu")
    assert st == 0
    check(x, o, S, cache, reference(x, "silu"))
