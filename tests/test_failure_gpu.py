"""Failure detection without a GPU fault.

Every wait in the prefill kernel is bounded.  The test hook kda_debug_stall_next_prefill
makes the prep warps withhold one hand-off (a flag that nothing then sets) and shortens
the waits; the recurrence's wait runs out, both warp groups leave their loops together,
copies and tensor-core products in flight land, the tensor memory is released, and the
host reads KDA_ERR_TIMEOUT from dev_status.  The context stays usable: the next call on
the same stream returns the oracle's result."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu
TIMEOUT = 6


def call(d, st):
    return kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S_in=d["S0"], dev_status=st)


@pytest.mark.parametrize("chunk", [0, 3])
def test_withheld_handoff_times_out_and_the_context_survives(chunk):
    inp = inputs.make_prefill([640, 300], H=2, seed=95, device="cpu", s0_std=0.02)
    d = to_device(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.debug_stall_next_prefill(chunk)
    call(d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == TIMEOUT
    # the next call is unaffected (the hook is one-shot) and exact to the path's tolerance
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, S, _ = call(d, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = oracle_units(inp, [(s, h) for s in range(2) for h in range(2)])
    cu = inp.cu_seqlens.tolist()
    og = np.concatenate([host(o[cu[s]:cu[s + 1], h]) for (s, h) in ref])
    assert rel_max(og, np.concatenate([r["o"] for r in ref.values()])) <= O_TOL
    assert rel_fro(np.stack([host(S[s, h]) for (s, h) in ref]), np.stack([r["S"] for r in ref.values()])) <= S_TOL
