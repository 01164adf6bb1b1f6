"""kda_prefill_noalloc: the prefill variant for callers that cannot allocate device memory
(for example a plugin whose host framework owns all device memory and hands it only input
and output tensors).  It must give what kda_prefill gives, using the library's own fixed
scratch array instead of a caller workspace, call after call.

This file sorts last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process."""
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu


def _case(seed, lengths, H):
    x = inputs.make_prefill(lengths, H=H, seed=seed, device="cpu", decay="uniform", s0_std=0.02, ckpt_every=64)
    x.g.mul_(0.01)  # slow decay, so the split's transition matrices matter
    return to_device(x)


def _both(d, n_segments):
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"])
    kw = dict(S_in=d["S0"], ckpt_off=d["ckpt_off"], ckpt_pos=d["ckpt_pos"], n_segments=n_segments)
    ref = kda.prefill(*args, **kw)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = kda.prefill_noalloc(*args, dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ref, got


def _close(ref, got):
    (o_r, S_r, c_r), (o_g, S_g, c_g) = ref, got
    assert rel_max(host(o_g), host(o_r)) <= O_TOL
    assert rel_fro(host(S_g), host(S_r)) <= S_TOL
    assert rel_fro(host(c_g), host(c_r)) <= S_TOL


def test_noalloc_matches_prefill_on_two_calls_in_a_row():
    # two different split problems back to back: the second call reuses the scratch the
    # first one left behind
    a = _case(401, [3000, 700], H=3)
    _close(*_both(a, n_segments=4))
    b = _case(402, [1900], H=2)
    _close(*_both(b, n_segments=3))


def test_noalloc_without_split_needs_no_scratch():
    c = _case(403, [500, 64], H=2)
    _close(*_both(c, n_segments=1))


def test_noalloc_rejects_a_problem_larger_than_its_scratch():
    d = _case(404, [8192], H=16)  # 64 forced segments x 16 heads needs ~200 MB of scratch
    assert kda.prefill_workspace_size(1, 16, 8192, n_segments=64) > kda.NOALLOC_SCRATCH_BYTES
    with pytest.raises(kda.KdaError) as e:
        kda.prefill_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], n_segments=64)
    assert e.value.status == 4  # KDA_ERR_WORKSPACE
