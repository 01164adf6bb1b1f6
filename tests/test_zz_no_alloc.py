"""kda_prefill_noalloc: the prefill variant for callers that cannot allocate device memory
(for example a plugin whose host framework owns all device memory and hands it only input
and output tensors).  It runs the same kernels on the same plan as kda_prefill, with the
split path's scratch taken from the library's own fixed array instead of a caller
workspace, so its outputs must equal kda_prefill's bit for bit, call after call (a stale
scratch entry left by an earlier call would change bits); one case is also checked
against the oracle.

This file sorts last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process."""
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu


def _case(seed, lengths, H, scale=0.01):
    x = inputs.make_prefill(lengths, H=H, seed=seed, device="cpu", decay="uniform", s0_std=0.02, ckpt_every=64)
    x.g.mul_(scale)  # slow decay, so the split's transition matrices matter
    return x


def _both(d, n_segments):
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    kw = dict(S_in=d["S0"], ckpt_off=d["ckpt_off"], ckpt_pos=d["ckpt_pos"], n_segments=n_segments)
    ref = kda.prefill(*args, **kw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = kda.prefill_noalloc(*args, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ref, got


def _same(ref, got):
    for r, g in zip(ref, got):
        assert torch.equal(r, g)


def test_noalloc_equals_prefill_bitwise_on_two_calls_in_a_row():
    # two different split problems back to back: the second call reuses the scratch the
    # first one left behind
    a = to_device(_case(401, [3000, 700], H=3))
    _same(*_both(a, n_segments=4))
    b = to_device(_case(402, [1900], H=2))
    _same(*_both(b, n_segments=3))
    _same(*_both(a, n_segments=4))  # and the first problem again, over the second's leftovers


def test_noalloc_with_the_automatic_split_against_the_oracle():
    # n_segments = 0: the library's own rule splits these sequences (2 heads, 20000 tokens)
    x = _case(405, [20000, 300], H=2)
    assert kda.prefill_workspace_size(2, 2, 20300) > 0
    d = to_device(x)
    ref, got = _both(d, n_segments=0)
    _same(ref, got)
    o, S, ck = got
    units = [(s, h) for s in range(2) for h in range(2)]
    orc = oracle_units(x, units)
    cu = x.cu_seqlens.tolist()
    off = x.ckpt_off.tolist()
    import numpy as np
    og = np.concatenate([host(o[cu[s]:cu[s + 1], h]) for s, h in units])
    orf = np.concatenate([orc[(s, h)]["o"] for s, h in units])
    assert rel_max(og, orf) <= O_TOL
    assert rel_fro(np.stack([host(S[s, h]) for s, h in units]), np.stack([orc[u]["S"] for u in units])) <= S_TOL
    for s, h in units:
        assert rel_fro(host(ck[off[s]:off[s + 1], h]), orc[(s, h)]["ckpts"]) <= S_TOL


def test_noalloc_without_split_needs_no_scratch():
    c = to_device(_case(403, [500, 64], H=2))
    _same(*_both(c, n_segments=1))


def test_noalloc_scratch_holds_the_long_workload():
    # the 1M-token, 8-head prefill with the library's own split fits the built-in scratch on
    # this device (the plan depends on its SM count)
    assert 0 < kda.prefill_workspace_size(1, 8, 1 << 20, n_segments=0) <= kda.NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    d = to_device(_case(404, [8192], H=16))  # 64 forced segments x 16 heads needs ~200 MB of scratch
    assert kda.prefill_workspace_size(1, 16, 8192, n_segments=64) > kda.NOALLOC_SCRATCH_BYTES
    with pytest.raises(kda.KdaError) as e:
        kda.prefill_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], n_segments=64)
    assert e.value.status == 4  # KDA_ERR_WORKSPACE
