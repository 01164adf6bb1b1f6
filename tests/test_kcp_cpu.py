"""Cross-device KCP's exchange (``kimi_delta_attention_prefill_gb300.kcp``) on CPU ranks:
3 processes, gloo on 127.0.0.1, with the fp64 oracle standing in for the device parts
(``oracle.segments``: the pair (M, S~) of a token range, its fold onto an entry state; the
oracle's recurrence for the second pass).  "部署 Kimi K3 ..." section 2.

  * the ranks' outputs, put back in token order, equal the unsplit recurrence (sequences
    cut unevenly, one rank holding no rows of one sequence, nonzero entry states);
  * a rank whose device part raises makes every rank raise KcpError before the exchange;
  * a rank that never arrives makes the others raise KcpError once the time limit runs
    out: no hang, no collective entered."""
import datetime
import multiprocessing as mp
import os
import socket
import sys
import time

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LENS = [300, 120]                       # two sequences
CUTS = [[0, 100, 220, 300], [0, 70, 70, 120]]  # rank r holds rows [cut[r], cut[r + 1]) of each
H, SEED = 2, 77


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _full():
    from kimi_delta_attention_prefill_gb300 import inputs
    return inputs.make_prefill(LENS, H=H, seed=SEED, device="cpu", decay="uniform", s0_std=0.02)


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _local(x, rank):
    """This rank's rows of every sequence, packed, as numpy (bf16 bits for q, k, v)."""
    cu = x.cu_seqlens.tolist()
    rows = np.concatenate([np.arange(cu[s] + CUTS[s][rank], cu[s] + CUTS[s][rank + 1]) for s in range(len(LENS))])
    lens = [CUTS[s][rank + 1] - CUTS[s][rank] for s in range(len(LENS))]
    loc = {n: getattr(x, n)[rows] for n in ("q", "k", "v", "g", "beta")}
    return {"q": _bits(loc["q"]), "k": _bits(loc["k"]), "v": _bits(loc["v"]), "g": loc["g"].numpy(),
            "beta": loc["beta"].numpy(), "cu": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)}


def oracle_parts(fail=False):
    import torch
    import oracle
    from oracle import segments as seg
    from kimi_delta_attention_prefill_gb300.kcp import DeviceParts
    bf = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    def pairs(x):
        if fail:
            raise RuntimeError("injected device failure")
        cu = x["cu"]
        N = cu.shape[0] - 1
        M = np.zeros((N, H, 128, 128))
        St = np.zeros((N, H, 128, 128))
        for s in range(N):
            a, b = int(cu[s]), int(cu[s + 1])
            for h in range(H):
                M[s, h] = seg.transition(bf(x["k"][a:b, h]), x["g"][a:b, h], x["beta"][a:b, h]) if b > a else np.eye(128)
            if b > a:
                r = oracle.prefill(x["q"][a:b], x["k"][a:b], x["v"][a:b], x["g"][a:b], x["beta"][a:b],
                                   np.array([0, b - a], np.int32), want_o=False)
                St[s] = r["S_out"][0]
        return torch.from_numpy(M), torch.from_numpy(St)

    def combine(Ms, Sts, S_in):
        E = np.zeros(Ms.shape[1:]) if S_in is None else np.array(S_in, np.float64)
        for s in range(E.shape[0]):
            for h in range(E.shape[1]):
                _, E[s, h] = seg.entry_states([(Ms[r, s, h].numpy(), Sts[r, s, h].numpy()) for r in range(Ms.shape[0])],
                                              E[s, h])
        return torch.from_numpy(E)

    def run(x, entry):
        r = oracle.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], S_in=entry.numpy())
        return r["o"], r["S_out"]

    return DeviceParts(pairs, combine, run)


def _rank(rank, world, port, scenario, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    store = dist.TCPStore("127.0.0.1", port, world, rank == 0, timeout=datetime.timedelta(seconds=60))
    dist.init_process_group("gloo", store=dist.PrefixStore("pg", store), rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=30))
    from kimi_delta_attention_prefill_gb300.kcp import KcpError, kcp_prefill
    x = _full()
    if scenario == "absent" and rank == 1:
        out.put((rank, "absent", None))
        time.sleep(8)  # alive (so rank 0's store stays up for everyone) but never posts
        return
    parts = oracle_parts(fail=(scenario == "fail" and rank == 1))
    t0 = time.monotonic()
    try:
        o, S = kcp_prefill(_local(x, rank), x.S0.double(), store, parts=parts,
                           timeout_s=2.0 if scenario == "absent" else 60.0)
        out.put((rank, "ok", (o, S)))
    except KcpError as e:
        out.put((rank, "kcp_error", (str(e), time.monotonic() - t0)))
    if scenario == "ok":
        dist.destroy_process_group()


def _run(scenario, world=3):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, scenario, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        r, kind, payload = out.get(timeout=180)
        got[r] = (kind, payload)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


def test_kcp_three_ranks_equal_the_unsplit_recurrence():
    import oracle
    got = _run("ok")
    assert all(k == "ok" for k, _ in got.values()), got
    x = _full()
    ref = oracle.prefill(_bits(x.q), _bits(x.k), _bits(x.v), x.g.numpy(), x.beta.numpy(), x.cu_seqlens.numpy(),
                         S_in=x.S0.numpy())
    cu = x.cu_seqlens.tolist()
    for s in range(len(LENS)):
        o = np.concatenate([got[r][1][0][int(sum(CUTS[t][r + 1] - CUTS[t][r] for t in range(s))):][
            :CUTS[s][r + 1] - CUTS[s][r]] for r in range(3)])
        o_ref = ref["o"][cu[s]:cu[s + 1]]
        assert np.abs(o - o_ref).max() <= 1e-5 * np.abs(o_ref).max()
        S_last = got[2][1][1][s]
        assert np.linalg.norm(S_last - ref["S_out"][s]) <= 1e-6 * np.linalg.norm(ref["S_out"][s])


def test_kcp_failed_rank_stops_every_rank_before_the_exchange():
    got = _run("fail")
    assert {r: k for r, (k, _) in got.items()} == {0: "kcp_error", 1: "kcp_error", 2: "kcp_error"}
    assert "[1] failed" in got[0][1][0] and "[1] failed" in got[2][1][0]
    assert "injected device failure" in got[1][1][0]
    assert got[1][1][1] < 5.0  # the failed rank left at once


def test_kcp_missing_rank_ends_the_call_after_the_time_limit():
    got = _run("absent")
    assert got[1][0] == "absent"
    for r in (0, 2):
        kind, (msg, dt) = got[r]
        assert kind == "kcp_error" and "did not post" in msg and "[1]" in msg
        assert 1.5 <= dt <= 20.0
