"""kda_prefill_host (host buffers, pipelined transfers) on the GPU.

The blocks go through the chunks and fp32 states of one device call, so the host call's o
and final states equal kda_prefill's on the same inputs bit for bit (no sequence split into
segments at these sizes); one case is also checked against the fp64 oracle directly."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu


def device_call(inp):
    d = to_device(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, S, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S_in=d["S0"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o.cpu(), S.cpu()


def host_call(inp, block=0):
    pin = lambda t: None if t is None else t.contiguous().pin_memory()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, S = kda.prefill_host(pin(inp.q), pin(inp.k), pin(inp.v), pin(inp.g), pin(inp.beta),
                            inp.cu_seqlens.to(torch.int32).contiguous(), S_in=pin(inp.S0), block_tokens=block,
                            dev_status=st)
    torch.cuda.current_stream().synchronize()
    assert int(st.item()) == 0
    return o, S


@pytest.mark.parametrize("block", [0, 64, 256])
def test_packed_equals_device_call(block):
    lens = [5, 64, 1, 300, 0, 130, 700]
    inp = inputs.make_prefill(lens, H=3, seed=91, device="cpu", s0_std=0.02, decay="uniform")
    o_ref, S_ref = device_call(inp)
    o, S = host_call(inp, block)
    assert torch.equal(o, o_ref)
    assert torch.equal(S, S_ref)


def test_single_long_sequence_default_blocks():
    inp = inputs.make_prefill([8192], H=8, seed=92, device="cpu")
    o_ref, S_ref = device_call(inp)
    assert len(kda.prefill_host_blocks(inp.cu_seqlens.to(torch.int32))) == 10  # 8 x 1024, the last split 768 + 256
    o, S = host_call(inp)
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)


def test_against_the_oracle():
    lens = [200, 77]
    inp = inputs.make_prefill(lens, H=2, seed=93, device="cpu", s0_std=0.02)
    o, S = host_call(inp, 64)
    ref = oracle_units(inp, [(s, h) for s in range(2) for h in range(2)])
    cu = inp.cu_seqlens.tolist()
    og = np.concatenate([host(o[cu[s]:cu[s + 1], h]) for (s, h) in ref])
    orf = np.concatenate([r["o"] for r in ref.values()])
    assert rel_max(og, orf) <= O_TOL
    assert rel_fro(np.stack([host(S[s, h]) for (s, h) in ref]), np.stack([r["S"] for r in ref.values()])) <= S_TOL


def test_all_empty_sequences_copy_the_state():
    inp = inputs.make_prefill([0, 0, 0], H=2, seed=94, device="cpu", s0_std=0.02)
    o, S = host_call(inp)
    assert torch.equal(S, inp.S0)
