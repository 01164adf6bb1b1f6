"""Cross-device KCP's device parts on one GPU ("部署 Kimi K3 ..." section 2), through the C ABI:

  * kda_prefill_pairs: the pair (M, S~) of each (sequence, head) against the oracle's
    literal transition product and its zero-entry state (the state bar, 1e-3 relative
    Frobenius); a sequence with no rows gives exactly (I, 0);
  * kda_combine_pairs: the fold E = S~_r + M_r E against numpy, fp32;
  * the ranks' device parts run one after another on this GPU (pairs of every rank, each
    rank's combine of the pairs before it, its prefill from the true entry state), and,
    through kcp.kcp_prefill on a one-rank group, the library's device parts: the
    outputs in token order against the unsplit oracle run (o bar 1e-2, state bar 1e-3)."""
import datetime

import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu
CUTS = [[0, 1000, 2100, 3000], [0, 64, 64, 500]]  # three ranks' rows of two sequences
LENS = [c[-1] for c in CUTS]


def _full():
    x = inputs.make_prefill(LENS, H=2, seed=91, device="cpu", decay="uniform", s0_std=0.02)
    x.g.mul_(0.004)  # slow decay: the transitions stay far from zero
    return x


def _rank_rows(x, r):
    cu = x.cu_seqlens.tolist()
    rows = torch.cat([torch.arange(cu[s] + CUTS[s][r], cu[s] + CUTS[s][r + 1]) for s in range(len(LENS))])
    lens = [CUTS[s][r + 1] - CUTS[s][r] for s in range(len(LENS))]
    part = inputs.PrefillInputs(x.q[rows], x.k[rows], x.v[rows], x.g[rows], x.beta[rows], None,
                                torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32))
    return part, to_device(part)


def test_pairs_against_the_oracle():
    """The pair of a 150-row range (where M stays far from 0 and from I) and of an empty one.
    M is a contraction (||M||_2 <= 1), so its error is judged by what it does to an exit
    state: ||M - M_ref||_F <= 1e-3 bounds the exit state's error by 1e-3 of the entry
    state's norm; S~ within the state bar."""
    import oracle
    from oracle import segments as seg
    x = inputs.make_prefill([150, 0], H=2, seed=93, device="cpu", decay="uniform")  # S~: zero entry state
    x.g.mul_(0.004)
    d = to_device(x)
    M, St = kda.prefill_pairs(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    torch.cuda.synchronize()
    bf = lambda t: t.float().double().numpy()
    ref = oracle_units(x, [(0, 0), (0, 1)])
    for h in range(2):
        Mref = seg.transition(bf(x.k[:, h]), x.g[:, h].double().numpy(), x.beta[:, h].double().numpy())
        assert 0.1 < np.linalg.norm(Mref, 2) <= 1.0 + 1e-9 and np.abs(Mref - np.eye(128)).max() > 0.1
        assert np.linalg.norm(host(M[0, h]) - Mref) <= S_TOL
        assert rel_fro(host(St[0, h]), ref[(0, h)]["S"]) <= S_TOL
    assert torch.equal(M[1], torch.eye(128, device="cuda").expand(2, 128, 128))
    assert torch.equal(St[1], torch.zeros_like(St[1]))


def test_pairs_at_full_width_equal_a_narrow_launch_bit_for_bit():
    """Pair mode with at least one CTA per SM (the compact kernel instance) against the same
    heads in a narrow launch (the full instance): the same arithmetic, so the same bits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = (sms + 3) // 4 + 2  # 2 sequences x 2 items x H >= SMs
    x = inputs.make_prefill([150, 70], H=H, seed=94, device="cpu", decay="uniform")
    x.g.mul_(0.004)
    d = to_device(x)
    M, St = kda.prefill_pairs(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    narrow = {key: (val[:, :2].contiguous() if key in ("q", "k", "v", "g", "beta") else val) for key, val in d.items()}
    M2, St2 = kda.prefill_pairs(narrow["q"], narrow["k"], narrow["v"], narrow["g"], narrow["beta"],
                                narrow["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(M[:, :2], M2) and torch.equal(St[:, :2], St2)
    ref = oracle_units(x, [(0, H - 1), (1, H - 1)])
    for s in range(2):
        assert rel_fro(host(St[s, H - 1]), ref[(s, H - 1)]["S"]) <= S_TOL


def test_combine_against_numpy():
    gen = torch.Generator().manual_seed(5)
    R, N, H = 3, 2, 3
    M = (torch.randn((R, N, H, 128, 128), generator=gen) * 0.05 + torch.eye(128) * 0.9).float()
    St = torch.randn((R, N, H, 128, 128), generator=gen).float()
    S_in = torch.randn((N, H, 128, 128), generator=gen).float()
    E = kda.combine_pairs(M.cuda(), St.cuda(), S_in=S_in.cuda())
    E0 = kda.combine_pairs(M[:0].cuda(), St[:0].cuda(), S_in=None)
    torch.cuda.synchronize()
    ref = S_in.double()
    for r in range(R):
        ref = St[r].double() + M[r].double() @ ref
    assert rel_fro(host(E), ref.numpy()) <= 1e-5
    assert torch.equal(E0, torch.zeros_like(E0))


def _check(x, outs, S_last):
    ref = oracle_units(x, [(s, h) for s in range(2) for h in range(2)])
    cu = x.cu_seqlens.tolist()
    og, orf = [], []
    for s in range(2):
        for h in range(2):
            rows = []
            for r in range(3):
                o_r, cu_r = outs[r]
                rows.append(host(o_r[cu_r[s]:cu_r[s + 1], h]))
            og.append(np.concatenate(rows))
            orf.append(ref[(s, h)]["o"])
    assert rel_max(np.concatenate(og), np.concatenate(orf)) <= O_TOL
    assert rel_fro(np.stack([host(S_last[s, h]) for s in range(2) for h in range(2)]),
                   np.stack([ref[(s, h)]["S"] for s in range(2) for h in range(2)])) <= S_TOL


def test_three_ranks_one_after_another_equal_the_unsplit_run():
    x = _full()
    S_in = x.S0.cuda()
    parts = [_rank_rows(x, r) for r in range(3)]
    pairs = [kda.prefill_pairs(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"]) for _, d in parts]
    Ms = torch.stack([p[0] for p in pairs])
    Sts = torch.stack([p[1] for p in pairs])
    outs, S = [], None
    for r, (part, d) in enumerate(parts):
        entry = kda.combine_pairs(Ms[:r].contiguous(), Sts[:r].contiguous(), S_in=S_in)
        o, S, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S_in=entry)
        outs.append((o, part.cu_seqlens.tolist()))
    torch.cuda.synchronize()
    _check(x, outs, S)


def test_kcp_prefill_on_a_one_rank_group_uses_the_library():
    import torch.distributed as dist
    from kimi_delta_attention_prefill_gb300.kcp import kcp_prefill
    store = dist.HashStore()
    dist.init_process_group("gloo", store=store, rank=0, world_size=1, timeout=datetime.timedelta(seconds=30))
    try:
        x = inputs.make_prefill([700], H=2, seed=92, device="cpu", s0_std=0.02)
        d = to_device(x)
        o, S, _ = kcp_prefill(d, d["S0"], store, timeout_s=10.0)
        torch.cuda.synchronize()
        ref = oracle_units(x, [(0, 0), (0, 1)])
        assert rel_max(np.stack([host(o[:, h]) for h in range(2)]), np.stack([ref[(0, h)]["o"] for h in range(2)])) <= O_TOL
        assert rel_fro(np.stack([host(S[0, h]) for h in range(2)]), np.stack([ref[(0, h)]["S"] for h in range(2)])) <= S_TOL
    finally:
        dist.destroy_process_group()
