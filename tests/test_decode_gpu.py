"""Decode / verify kernel against the fp64 oracle (fp32 tolerance 1e-4), through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import DECODE_TOL, bits, host, rel_max

pytestmark = pytest.mark.gpu


def run_case(B, n_tok, H, seed, commit="all", n_commit=None):
    x = inputs.make_decode(B, n_tok, H, seed=seed, device="cuda", commit=commit)
    if n_commit is not None:
        x.n_commit = torch.tensor(n_commit, dtype=torch.int32)
    S = x.S0.clone()
    nc = None if x.n_commit is None else x.n_commit.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.decode(x.q, x.k, x.v, x.g, x.beta, S, n_commit=nc, dev_status=status)
    torch.cuda.synchronize()
    ref = oracle.decode(bits(x.q), bits(x.k), bits(x.v), host(x.g), host(x.beta), host(x.S0),
                        None if x.n_commit is None else x.n_commit.numpy())
    return x, o, S, ref, int(status.item())


@pytest.mark.parametrize("n_tok", [1, 2, 3, 4])
@pytest.mark.parametrize("commit", ["all", "random"])
def test_decode_small(n_tok, commit):
    x, o, S, ref, st = run_case(B=7, n_tok=n_tok, H=5, seed=10 + n_tok, commit=commit)
    assert st == 0
    assert rel_max(host(o), ref["o"]) <= DECODE_TOL
    assert rel_max(host(S), ref["S"]) <= DECODE_TOL


def test_decode_commit_zero_leaves_state_bitwise():
    x, o, S, ref, st = run_case(B=4, n_tok=4, H=3, seed=21, n_commit=[0, 4, 0, 2])
    assert st == 0
    assert torch.equal(S[0], x.S0[0]) and torch.equal(S[2], x.S0[2])
    assert rel_max(host(S), ref["S"]) <= DECODE_TOL
    assert rel_max(host(o), ref["o"]) <= DECODE_TOL


def test_decode_bad_commit_reports_and_skips():
    x = inputs.make_decode(3, 2, 2, seed=22, device="cuda")
    S = x.S0.clone()
    nc = torch.tensor([1, 3, -1], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.decode(x.q, x.k, x.v, x.g, x.beta, S, n_commit=nc, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 7  # KDA_ERR_DEVICE_CHECK
    assert torch.equal(S[1], x.S0[1]) and torch.equal(S[2], x.S0[2])
    assert not torch.equal(S[0], x.S0[0])


def test_decode_empty_batch_is_noop():
    x = inputs.make_decode(2, 1, 2, seed=23, device="cuda")
    q = x.q[:0]
    o = kda.decode(q, x.k[:0], x.v[:0], x.g[:0], x.beta[:0], x.S0[:0])
    assert o.shape == (0, 1, 2, 128)


@pytest.mark.parametrize("name", ["decode", "verify"])
def test_decode_full_size(name):
    """The 256 x 96 decode step and the 4-token verify with random commits, every unit."""
    w = inputs.WORKLOADS[name]
    x = inputs.make_workload(name, device="cuda")
    S = x.S0.clone()
    nc = None if x.n_commit is None else x.n_commit.cuda()
    o = kda.decode(x.q, x.k, x.v, x.g, x.beta, S, n_commit=nc)
    torch.cuda.synchronize()
    ref = oracle.decode(bits(x.q), bits(x.k), bits(x.v), host(x.g), host(x.beta), host(x.S0),
                        None if x.n_commit is None else x.n_commit.numpy())
    assert o.shape == (w["B"], w["n_tok"], w["H"], 128)
    assert rel_max(host(o), ref["o"]) <= DECODE_TOL
    assert rel_max(host(S), ref["S"]) <= DECODE_TOL
