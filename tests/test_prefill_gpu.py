"""Chunkwise prefill kernel against the fp64 oracle, through the C ABI.

Bar: o within max|o - o_ref| / max|o_ref| <= 1e-2; final state and each checkpoint within
relative Frobenius error <= 1e-3; checkpoint positions and varlen boundaries bit-exact
(packed == standalone bit for bit; the checkpoint at len equals S_out bit for bit; no write
outside a sequence's rows)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu


def run_gpu(inp, n_segments=0, o_pad=0):
    d = to_device(inp)
    T, H = inp.q.shape[0], inp.q.shape[1]
    o_buf = torch.full((T + 2 * o_pad, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = o_buf[o_pad:o_pad + T]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, S, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S_in=d["S0"],
                           ckpt_off=d["ckpt_off"], ckpt_pos=d["ckpt_pos"], o=o, n_segments=n_segments,
                           dev_status=status)
    torch.cuda.synchronize()
    return o, S, ck, int(status.item()), o_buf


def check_against_oracle(inp, o, S, ck, units=None, o_stride=1):
    n_seq, H = inp.n_seq, inp.q.shape[1]
    units = units or [(s, h) for s in range(n_seq) for h in range(H)]
    ref = oracle_units(inp, units, o_stride=o_stride)
    cu = inp.cu_seqlens.tolist()
    og, orf, sg, srf, cg, crf = [], [], [], [], [], []
    for (s, h), r in ref.items():
        a, b = cu[s], cu[s + 1]
        og.append(host(o[a:b:o_stride, h]))
        orf.append(r["o"])
        sg.append(host(S[s, h]))
        srf.append(r["S"])
        if ck is not None and r["ckpts"] is not None and r["ckpts"].shape[0]:
            lo, hi = int(inp.ckpt_off[s]), int(inp.ckpt_off[s + 1])
            cg.append(host(ck[lo:hi, h]))
            crf.append(r["ckpts"])
    og, orf = np.concatenate(og), np.concatenate(orf)
    e_o = rel_max(og, orf) if orf.size else 0.0
    e_s = rel_fro(np.stack(sg), np.stack(srf))
    assert e_o <= O_TOL, f"o error {e_o:.3e}"
    assert e_s <= S_TOL, f"state error {e_s:.3e}"
    for a_, b_ in zip(cg, crf):
        assert rel_fro(a_, b_) <= S_TOL
    return e_o, e_s


def test_tiny_config():
    inp = inputs.make_workload("tiny", device="cpu")
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck)


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 200, 257])
@pytest.mark.parametrize("decay", ["sigmoid", "uniform"])
def test_single_sequence_shapes(T, decay):
    inp = inputs.make_prefill([T], H=3, seed=100 + T, device="cpu", decay=decay, s0_std=0.02)
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck)


def test_zero_initial_state_and_all_g_at_floor():
    inp = inputs.make_prefill([300], H=2, seed=7, device="cpu", decay="uniform")
    inp.g.fill_(inputs.G_MIN)  # every step at the decay floor: the rebasing's worst case
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
    check_against_oracle(inp, o, S, ck)


def test_weak_decay_long_memory():
    inp = inputs.make_prefill([1024], H=2, seed=8, device="cpu", decay="uniform", s0_std=0.02)
    inp.g.mul_(0.002)  # g in [-0.01, 0): the state remembers hundreds of tokens
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck)


def _varlen_small():
    lens = [5, 64, 1, 130, 0, 77, 192, 64]
    inp = inputs.make_prefill(lens, H=4, seed=31, device="cpu", decay="uniform", s0_std=0.02)
    off, pos = [0], []
    for n in lens:
        p = sorted(set(list(range(64, n + 1, 64)) + ([n] if n > 0 else [])))
        pos += p
        off.append(len(pos))
    inp.ckpt_off = torch.tensor(off, dtype=torch.int32)
    inp.ckpt_pos = torch.tensor(pos, dtype=torch.int32)
    return inp


def test_varlen_checkpoints_and_boundaries():
    inp = _varlen_small()
    o, S, ck, st, o_buf = run_gpu(inp, o_pad=64)
    assert st == 0
    check_against_oracle(inp, o, S, ck)
    # no write outside the packed rows
    assert torch.isnan(o_buf[:64].float()).all() and torch.isnan(o_buf[-64:].float()).all()
    assert not torch.isnan(o.float()).any()
    cu = inp.cu_seqlens.tolist()
    off = inp.ckpt_off.tolist()
    pos = inp.ckpt_pos.tolist()
    for s in range(inp.n_seq):
        a, b = cu[s], cu[s + 1]
        # the checkpoint at p = len is the final state, bit for bit
        if b > a:
            assert pos[off[s + 1] - 1] == b - a
            assert torch.equal(ck[off[s + 1] - 1], S[s])
        # packed == standalone, bit for bit
        one = inputs.PrefillInputs(inp.q[a:b], inp.k[a:b], inp.v[a:b], inp.g[a:b], inp.beta[a:b],
                                   inp.S0[s:s + 1], torch.tensor([0, b - a], dtype=torch.int32),
                                   torch.tensor([0, off[s + 1] - off[s]], dtype=torch.int32),
                                   torch.tensor(pos[off[s]:off[s + 1]], dtype=torch.int32))
        o1, S1, ck1, st1, _ = run_gpu(one)
        assert st1 == 0
        assert torch.equal(o1, o[a:b])
        assert torch.equal(S1[0], S[s])
        if off[s + 1] > off[s]:
            assert torch.equal(ck1, ck[off[s]:off[s + 1]])


def test_restart_from_checkpoint_2560():
    """Resume at 2560 = 5 x 512 from the checkpoint the kernel wrote; the rest of the run
    matches the continuous one (bitwise: no segment split)."""
    T, P = 2800, 2560
    inp = inputs.make_prefill([T], H=2, seed=41, device="cpu", decay="sigmoid", s0_std=0.02, ckpt_every=512)
    o, S, ck, st, _ = run_gpu(inp, n_segments=1)
    assert st == 0
    assert inp.ckpt_pos.tolist() == [512, 1024, 1536, 2048, 2560]
    tail = inputs.PrefillInputs(inp.q[P:], inp.k[P:], inp.v[P:], inp.g[P:], inp.beta[P:],
                                ck[4:5].cpu(), torch.tensor([0, T - P], dtype=torch.int32))
    o2, S2, _, st2, _ = run_gpu(tail, n_segments=1)
    assert st2 == 0
    assert torch.equal(o2, o[P:])
    assert torch.equal(S2, S)


def test_device_side_argument_checks():
    inp = inputs.make_prefill([64, 64], H=2, seed=5, device="cpu")
    bad = inputs.PrefillInputs(inp.q, inp.k, inp.v, inp.g, inp.beta, None,
                               torch.tensor([0, 100, 64], dtype=torch.int32))  # not monotone
    _, _, _, st, _ = run_gpu(bad)
    assert st == 7
    bad2 = inputs.PrefillInputs(inp.q, inp.k, inp.v, inp.g, inp.beta, None, inp.cu_seqlens,
                                torch.tensor([0, 1, 1], dtype=torch.int32), torch.tensor([30], dtype=torch.int32))
    _, _, _, st, _ = run_gpu(bad2)
    assert st == 7  # a checkpoint inside a chunk is not supported


def test_prefill_8k_full():
    """Model-width prefill (1 x 8192 tokens, 96 heads) in the benchmark's launch
    configuration: every head's final state and every row of o against the oracle."""
    inp = inputs.make_workload("prefill_8k", device="cuda")
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck)


def test_prefill_1m_sampled():
    """1M-token prefill on 8 heads through the planner's split: every head's final state
    against the oracle, and o on every 8th row of every head; every head finite."""
    inp = inputs.make_workload("prefill_1m", device="cuda")
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(S).all()
    check_against_oracle(inp, o, S, ck, units=[(0, h) for h in range(inp.q.shape[1])], o_stride=8)


def test_varlen_full_sampled():
    """64 packed sequences, 96 heads, stress decay, nonzero states, checkpoints every 512:
    one (sequence, head) unit of every sequence against the oracle (every row of o, the
    final state, every checkpoint), heads spread over the 96; every sequence's last
    checkpoint at len equals its final state bit for bit."""
    inp = inputs.make_workload("varlen", device="cuda")
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    H = inp.q.shape[1]
    rng = np.random.default_rng(0)
    units = [(s, int(h)) for s, h in zip(range(inp.n_seq), rng.integers(0, H, inp.n_seq))]
    check_against_oracle(inp, o, S, ck, units=units)
    off = inp.ckpt_off.tolist()
    for s in range(inp.n_seq):
        assert torch.equal(ck[off[s + 1] - 1], S[s]) or (inp.cu_seqlens[s + 1] - inp.cu_seqlens[s]) % 512 != 0


# ------------------------------------------------------------------ sequence split (P8)
def _weak(inp, scale):
    inp.g.mul_(scale)  # slow decay: the transition M of a segment stays far from zero
    return inp


@pytest.mark.parametrize("n_seg", [2, 3, 7])
@pytest.mark.parametrize("T", [1000, 2909])
def test_split_forced_segments(n_seg, T):
    inp = _weak(inputs.make_prefill([T], H=2, seed=200 + T + n_seg, device="cpu", decay="uniform", s0_std=0.02,
                                    ckpt_every=64), 0.004)
    o, S, ck, st, _ = run_gpu(inp, n_segments=n_seg)
    assert st == 0
    check_against_oracle(inp, o, S, ck)


def test_split_equals_unsplit_within_tolerance():
    inp = _weak(inputs.make_prefill([4096], H=3, seed=301, device="cpu", decay="uniform", s0_std=0.02), 0.002)
    o1, S1, _, st1, _ = run_gpu(inp, n_segments=1)
    o4, S4, _, st4, _ = run_gpu(inp, n_segments=4)
    assert st1 == 0 and st4 == 0
    from kda_gpu_util import rel_fro as rf, rel_max as rm
    assert rf(host(S4), host(S1)) <= S_TOL
    assert rm(host(o4), host(o1)) <= O_TOL
    check_against_oracle(inp, o4, S4, None)


def test_split_varlen_packed_equals_standalone():
    lens = [0, 1, 64, 65, 700, 1300]
    inp = _weak(inputs.make_prefill(lens, H=2, seed=302, device="cpu", decay="uniform", s0_std=0.02,
                                    ckpt_every=64), 0.01)
    o, S, ck, st, o_buf = run_gpu(inp, n_segments=5, o_pad=64)
    assert st == 0
    check_against_oracle(inp, o, S, ck)
    assert torch.isnan(o_buf[:64].float()).all() and torch.isnan(o_buf[-64:].float()).all()
    cu, off, pos = inp.cu_seqlens.tolist(), inp.ckpt_off.tolist(), inp.ckpt_pos.tolist()
    for s in range(inp.n_seq):
        a, b = cu[s], cu[s + 1]
        one = inputs.PrefillInputs(inp.q[a:b], inp.k[a:b], inp.v[a:b], inp.g[a:b], inp.beta[a:b],
                                   inp.S0[s:s + 1], torch.tensor([0, b - a], dtype=torch.int32),
                                   torch.tensor([0, off[s + 1] - off[s]], dtype=torch.int32),
                                   torch.tensor(pos[off[s]:off[s + 1]], dtype=torch.int32))
        o1, S1, ck1, st1, _ = run_gpu(one, n_segments=5)
        assert st1 == 0
        assert torch.equal(o1, o[a:b]) and torch.equal(S1[0], S[s])
        if off[s + 1] > off[s]:
            assert torch.equal(ck1, ck[off[s]:off[s + 1]])


def test_split_workspace_too_small_is_rejected():
    inp = inputs.make_prefill([3000], H=2, seed=303, device="cpu")
    d = to_device(inp)
    need = kda.prefill_workspace_size(1, 2, 3000, n_segments=3)
    assert need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], n_segments=3, workspace=ws)
    assert e.value.status == 4


def test_auto_planner_splits_few_heads_only():
    assert kda.prefill_workspace_size(1, 96, 8192) == 0
    assert kda.prefill_workspace_size(64, 96, 540672) == 0
    assert kda.prefill_workspace_size(1, 8, 1 << 20) > 0


@pytest.mark.parametrize("H,lens", [(1, [9000]), (130, [129, 64]), (7, [300, 1, 700])])
def test_head_counts(H, lens):
    """One head (a 9000-token sequence: two segments would not shorten the chain, so the
    planner keeps one), more heads than
    SMs (130: a grid wider than the GPU), and an odd count with packed sequences and
    checkpoints.  Every unit against the oracle for the small cases, sampled heads for 130."""
    inp = inputs.make_prefill(lens, H=H, seed=300 + H, device="cpu", s0_std=0.02, ckpt_every=64)
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    units = None if H < 100 else [(s, h) for s in range(len(lens)) for h in (0, 1, 64, 127, 129)]
    check_against_oracle(inp, o, S, ck, units=units)


@pytest.mark.parametrize("case", ["beta0", "beta1", "g0"])
def test_degenerate_gates(case):
    """beta = 0 (the state only decays: o_t = (e^{G_t} S0)^T q_t), beta = 1 (full delta-rule
    overwrite) and g = 0 (no decay at all, the rebasing's trivial case), packed, with
    checkpoints, against the oracle."""
    inp = inputs.make_prefill([200, 64, 130], H=2, seed=400, device="cpu", s0_std=0.02, ckpt_every=64)
    if case == "beta0":
        inp.beta.zero_()
    elif case == "beta1":
        inp.beta.fill_(1.0)
    else:
        inp.g.zero_()
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck)


# ------------------------------------------------------------ the delta rule's edge cases
def _exact_unit_keys(n, H, seed):
    """[n, H, 128] bf16 keys of norm exactly 1: +-1/8 on 64 random channels (64 / 64 = 1)."""
    gen = torch.Generator().manual_seed(seed)
    keys = torch.zeros(n, H, 128)
    for t in range(n):
        for h in range(H):
            idx = torch.randperm(128, generator=gen)[:64]
            keys[t, h, idx] = (torch.randint(0, 2, (64,), generator=gen).float() * 2 - 1) / 8
    keys = keys.to(torch.bfloat16)
    assert torch.equal((keys.double() ** 2).sum(-1), torch.ones(n, H, dtype=torch.float64))
    return keys


def test_repeated_identical_keys_beta1_no_decay():
    """Every token writes with the same unit key, beta = 1 and g = 0: L is all ones below the
    diagonal (the worst-conditioned (I + L) of the chunk form; INV = I minus the first
    subdiagonal) and each token replaces the key's whole component of the state
    ("Kimi K3 ... 服務性能" section 4: the delta rule overwrites along k).  Closed form with
    P = I - k k^T: S_t = P S_0 + k v_t^T and o_t = (P S_0)^T q_t + (k . q_t) v_t.  Several
    chunks and a ragged tail, against the oracle and the closed form."""
    T, H = 333, 2
    inp = inputs.make_prefill([T], H=H, seed=501, device="cpu", s0_std=0.02, ckpt_every=64)
    inp.k = _exact_unit_keys(1, H, 505).expand(T, H, 128).contiguous()
    inp.beta.fill_(1.0)
    inp.g.zero_()
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck)
    k = inp.k[0].double()                      # [H, d], exactly unit
    P = torch.eye(128, dtype=torch.float64) - torch.einsum("hi,hj->hij", k, k)
    PS0 = torch.einsum("hij,hjc->hic", P, inp.S0[0].double())
    q, v = inp.q.double(), inp.v.double()
    want = torch.einsum("hic,thi->thc", PS0, q) + torch.einsum("hi,thi->th", k, q)[..., None] * v
    assert rel_max(host(o), want.numpy()) <= O_TOL
    S_want = PS0 + torch.einsum("hi,hc->hic", k, v[-1])
    assert rel_fro(host(S[0]), S_want.numpy()) <= S_TOL


@pytest.mark.parametrize("decay", ["sigmoid", "uniform"])
def test_retrieval_invariant_unit_keys(decay):
    """Delta-rule retrieval ("Kimi K3.1 Pro 架构完全拆解" 3.1; "Kimi K3 ... 服務性能" 4): with
    beta = 1 and a unit key, S_t^T k_t = v_t right after the token, whatever the decay and
    the entry state.  With q = k the output is therefore o_t = v_t for every token.  The
    keys are exactly unit in bf16, so the invariant is exact; o against v within the o bar,
    and everything against the oracle."""
    T, H = 450, 3
    inp = inputs.make_prefill([T], H=H, seed=502, device="cpu", decay=decay, s0_std=0.02)
    inp.k = _exact_unit_keys(T, H, 503)
    inp.q = inp.k.clone()
    inp.beta.fill_(1.0)
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    assert rel_max(host(o), host(inp.v)) <= O_TOL
    check_against_oracle(inp, o, S, ck)


def test_large_values_within_the_fp16_operand_range():
    """The state path's operands are fp16 (largest finite value 65504): v scaled by 2^10
    (max |v| about 4.5e3) keeps the state, X and U well inside that range; every output
    against the oracle with the usual relative bars, and finite."""
    inp = inputs.make_prefill([700], H=2, seed=504, device="cpu", decay="sigmoid", s0_std=0.02, ckpt_every=64)
    inp.v = (inp.v.float() * 1024.0).to(torch.bfloat16)  # exact: a power of two
    inp.S0 = inp.S0 * 1024.0
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(S).all()
    check_against_oracle(inp, o, S, ck)


def _packed_equals_standalone(inp, o, S, ck, seqs):
    cu, off, pos = inp.cu_seqlens.tolist(), inp.ckpt_off.tolist(), inp.ckpt_pos.tolist()
    for s in seqs:
        a, b = cu[s], cu[s + 1]
        one = inputs.PrefillInputs(inp.q[a:b], inp.k[a:b], inp.v[a:b], inp.g[a:b], inp.beta[a:b],
                                   inp.S0[s:s + 1], torch.tensor([0, b - a], dtype=torch.int32),
                                   torch.tensor([0, off[s + 1] - off[s]], dtype=torch.int32),
                                   torch.tensor(pos[off[s]:off[s + 1]], dtype=torch.int32))
        o1, S1, ck1, st1, _ = run_gpu(one)
        assert st1 == 0
        assert torch.equal(o1, o[a:b]) and torch.equal(S1[0], S[s]), f"sequence {s}"
        if off[s + 1] > off[s]:
            assert torch.equal(ck1, ck[off[s]:off[s + 1]])


def test_full_gpu_packed_launch_longest_first_equals_standalone():
    """A packed launch with at least one unit per SM (the compact kernel instance, sequences
    taken longest first, ties by index) against the oracle and, bit for bit, against each
    sequence run alone (a few units: the full instance, launch order irrelevant)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = 4
    n_seq = (sms + H - 1) // H + 2
    rng = np.random.default_rng(404)
    lens = rng.integers(1, 700, size=n_seq).tolist()
    lens[3] = lens[7] = lens[11]  # ties in the ranking
    inp = inputs.make_prefill(lens, H=H, seed=404, device="cpu", decay="uniform", s0_std=0.02, ckpt_every=64)
    o, S, ck, st, o_buf = run_gpu(inp, o_pad=64)
    assert st == 0
    assert torch.isnan(o_buf[:64].float()).all() and torch.isnan(o_buf[-64:].float()).all()
    assert not torch.isnan(o.float()).any()
    units = [(s, h) for s in range(0, n_seq, 5) for h in range(H)]
    check_against_oracle(inp, o, S, ck, units=units)
    _packed_equals_standalone(inp, o, S, ck, range(n_seq))


@pytest.mark.parametrize("n_seq", [256, 257])
def test_ranking_limit_256_sequences(n_seq):
    """256 sequences: the largest launch that ranks them by length (each CTA compares 256 x
    256 lengths); 257: past the limit the packed launch keeps the index order.  Results do
    not depend on the order."""
    rng = np.random.default_rng(405)
    lens = rng.integers(1, 140, size=n_seq).tolist()
    inp = inputs.make_prefill(lens, H=1, seed=405, device="cpu", decay="uniform", s0_std=0.02, ckpt_every=64)
    o, S, ck, st, _ = run_gpu(inp)
    assert st == 0
    check_against_oracle(inp, o, S, ck, units=[(s, 0) for s in range(0, n_seq, 16)])
    _packed_equals_standalone(inp, o, S, ck, range(0, n_seq, 8))
