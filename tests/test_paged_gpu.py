"""Paged states (kda_prefill_paged, kda_decode_paged) through the C ABI.

"部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra 全景" section 3: each head's state is one
64 KiB block of a prefix cache, snapshotted at hash-aligned positions; a hit resumes from
the cached snapshot, which other requests may share, so it is read and never written
(copy on hit).  The paged entry points take every state through a page pool; the bar:
  * the same bits as the contiguous entry points on the same inputs (only addresses
    differ: o, final states and checkpoints bit for bit), and the oracle's tolerance on
    one case directly;
  * pages the call does not name as destinations are left bit-unchanged (canaries);
  * a call that would write a page twice, write a page another unit reads, or name a page
    outside the pool writes nothing and reports KDA_ERR_DEVICE_CHECK.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs
from kda_gpu_util import DECODE_TOL, O_TOL, S_TOL, host, oracle_units, rel_fro, rel_max, to_device

pytestmark = pytest.mark.gpu
DEVICE_CHECK = 7


def canary_pool(n_pages, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((n_pages, 128, 128), generator=gen, device="cuda")


def contiguous_prefill(inp, n_segments=0, gate=None, w=None):
    d = to_device(inp)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = {} if gate is None else dict(gate=gate.cuda(), norm_weight=None if w is None else w.cuda())
    o, S, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], S_in=d["S0"],
                           ckpt_off=d["ckpt_off"], ckpt_pos=d["ckpt_pos"], n_segments=n_segments, dev_status=st, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, S, ck


def paged_prefill(inp, pool, s_in, s_out, ck_page, n_segments=0, gate=None, w=None):
    d = to_device(inp)
    T, H, _ = inp.q.shape
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    kw = {} if gate is None else dict(gate=gate.cuda(), norm_weight=None if w is None else w.cuda())
    kda.prefill_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], pool,
                      s_in_page=None if s_in is None else s_in.cuda(),
                      s_out_page=None if s_out is None else s_out.cuda(), ckpt_off=d["ckpt_off"],
                      ckpt_pos=d["ckpt_pos"], ckpt_page=None if ck_page is None else ck_page.cuda(), o=o,
                      n_segments=n_segments, dev_status=st, **kw)
    torch.cuda.synchronize()
    return o, int(st.item())


def scatter_case(lens, H, seed, n_pages, ckpt_every=64, s0_std=0.02):
    inp = inputs.make_prefill(lens, H=H, seed=seed, device="cpu", s0_std=s0_std, ckpt_every=ckpt_every)
    n_units = len(lens) * H
    n_ck = 0 if inp.ckpt_pos is None else inp.ckpt_pos.shape[0] * H
    s_in, s_out, ck = inputs.make_page_tables([n_units, n_units, n_ck], n_pages, seed=seed)
    return inp, s_in, s_out, (ck if n_ck else None)


def load_entry_states(pool, inp, s_in):
    """The pool's entry pages hold the inputs' S0 (unit u = seq * H + h)."""
    n_seq, H = inp.S0.shape[0], inp.S0.shape[1]
    pool[s_in.long().cuda()] = inp.S0.reshape(n_seq * H, 128, 128).cuda()


@pytest.mark.parametrize("n_segments", [0, 3])
def test_prefill_paged_equals_contiguous(n_segments):
    lens = [5, 64, 1, 300, 0, 130]
    inp, s_in, s_out, ck = scatter_case(lens, H=3, seed=71, n_pages=256)
    pool = canary_pool(256, 1)
    load_entry_states(pool, inp, s_in)
    before = pool.clone()
    o_ref, S_ref, ck_ref = contiguous_prefill(inp, n_segments)
    o, st = paged_prefill(inp, pool, s_in, s_out, ck, n_segments)
    assert st == 0
    assert torch.equal(o, o_ref)
    H = 3
    assert torch.equal(pool[s_out.long()], S_ref.reshape(-1, 128, 128))
    assert torch.equal(pool[ck.long()], ck_ref.reshape(-1, 128, 128))
    untouched = torch.ones(256, dtype=torch.bool)
    untouched[s_out.long()] = False
    untouched[ck.long()] = False
    assert torch.equal(pool[untouched.cuda()], before[untouched.cuda()]), "a page outside the destinations changed"


def test_prefill_paged_gated_equals_contiguous():
    lens = [77, 200]
    inp, s_in, s_out, ck = scatter_case(lens, H=2, seed=72, n_pages=64)
    gate, w = inputs.make_output_stage(inp.q.shape[0], 2, seed=72)
    pool = canary_pool(64, 2)
    load_entry_states(pool, inp, s_in)
    o_ref, S_ref, ck_ref = contiguous_prefill(inp, gate=gate, w=w)
    o, st = paged_prefill(inp, pool, s_in, s_out, ck, gate=gate, w=w)
    assert st == 0
    assert torch.equal(o, o_ref)
    assert torch.equal(pool[s_out.long()], S_ref.reshape(-1, 128, 128))
    assert torch.equal(pool[ck.long()], ck_ref.reshape(-1, 128, 128))


def test_prefill_paged_against_the_oracle():
    """One paged call checked directly against the fp64 oracle (tolerances of the path)."""
    lens = [130, 64]
    inp, s_in, s_out, ck = scatter_case(lens, H=2, seed=73, n_pages=40)
    pool = canary_pool(40, 3)
    load_entry_states(pool, inp, s_in)
    o, st = paged_prefill(inp, pool, s_in, s_out, ck)
    assert st == 0
    ref = oracle_units(inp, [(s, h) for s in range(2) for h in range(2)])
    cu = inp.cu_seqlens.tolist()
    og, orf, sg, sr, cg, cr = [], [], [], [], [], []
    off = inp.ckpt_off.tolist()
    for (s, h), r in ref.items():
        og.append(host(o[cu[s]:cu[s + 1], h]))
        orf.append(r["o"])
        sg.append(host(pool[int(s_out[s * 2 + h])]))
        sr.append(r["S"])
        for j in range(off[s], off[s + 1]):
            cg.append(host(pool[int(ck[j * 2 + h])]))
        if r["ckpts"] is not None:
            cr.append(r["ckpts"])
    assert rel_max(np.concatenate(og), np.concatenate(orf)) <= O_TOL
    assert rel_fro(np.stack(sg), np.stack(sr)) <= S_TOL
    assert rel_fro(np.stack(cg), np.concatenate(cr)) <= S_TOL


def test_prefill_copy_on_hit_shared_snapshot():
    """Three sequences resume from one cached snapshot page: each continuation equals a
    contiguous run from that snapshot, and the snapshot page is bit-unchanged."""
    lens = [64, 129, 7]
    H = 2
    inp = inputs.make_prefill(lens, H=H, seed=74, device="cpu", s0_std=0.02)
    pool = canary_pool(32, 4)
    snap = [5, 9]  # one snapshot page per head, shared by all three sequences
    s_in = torch.tensor([snap[h] for s in range(3) for h in range(H)], dtype=torch.int32)
    s_out = torch.tensor([20 + u for u in range(3 * H)], dtype=torch.int32)
    shared = pool[snap].clone()
    inp.S0 = torch.stack([shared.cpu()] * 3)  # contiguous reference: every sequence starts from the snapshot
    o_ref, S_ref, _ = contiguous_prefill(inp)
    o, st = paged_prefill(inp, pool, s_in, s_out, None)
    assert st == 0
    assert torch.equal(o, o_ref)
    assert torch.equal(pool[s_out.long()], S_ref.reshape(-1, 128, 128))
    assert torch.equal(pool[snap], shared), "the shared snapshot was written"


def test_prefill_in_place_and_missing_pages():
    """s_out = s_in updates a unit's own page in place; -1 entries mean a zero entry state
    and no final-state write."""
    lens = [100, 64]
    H = 2
    inp = inputs.make_prefill(lens, H=H, seed=75, device="cpu", s0_std=0.02)
    pool = canary_pool(16, 5)
    s_in = torch.tensor([3, -1, 7, 11], dtype=torch.int32)
    s_out = torch.tensor([3, 12, 7, -1], dtype=torch.int32)
    S0 = torch.zeros(2, H, 128, 128)
    for u, pg in enumerate(s_in.tolist()):
        if pg >= 0:
            S0[u // H, u % H] = pool[pg].cpu()
    inp.S0 = S0
    before = pool.clone()
    o_ref, S_ref, _ = contiguous_prefill(inp)
    o, st = paged_prefill(inp, pool, s_in, s_out, None)
    assert st == 0 and torch.equal(o, o_ref)
    flat = S_ref.reshape(-1, 128, 128)
    assert torch.equal(pool[3], flat[0]) and torch.equal(pool[12], flat[1]) and torch.equal(pool[7], flat[2])
    keep = [p for p in range(16) if p not in (3, 12, 7)]
    assert torch.equal(pool[keep], before[keep])


@pytest.mark.parametrize("bad", ["dup_out", "write_shared_read", "ckpt_over_entry", "out_of_pool", "below_minus1"])
def test_prefill_page_violations_write_nothing(bad):
    lens = [64, 70]
    H = 2
    inp = inputs.make_prefill(lens, H=H, seed=76, device="cpu", s0_std=0.02, ckpt_every=64)
    n_ck = inp.ckpt_pos.shape[0]
    s_in = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    s_out = torch.tensor([4, 5, 6, 7], dtype=torch.int32)
    ck = torch.arange(8, 8 + n_ck * H, dtype=torch.int32)
    if bad == "dup_out":
        s_out[3] = 5
    elif bad == "write_shared_read":
        s_out[0] = 2  # unit 0 would overwrite unit 2's entry page
    elif bad == "ckpt_over_entry":
        ck[0] = 0  # sequence 0, head 0's first checkpoint over its own entry page
    elif bad == "out_of_pool":
        s_out[1] = 64
    else:
        s_in[2] = -2
    pool = canary_pool(64, 6)
    before = pool.clone()
    o, st = paged_prefill(inp, pool, s_in, s_out, ck)
    assert st == DEVICE_CHECK
    assert torch.isnan(o.float()).all(), "outputs were written"
    assert torch.equal(pool, before), "pages were written"


def decode_case(B, n_tok, H, seed, commit):
    x = inputs.make_decode(B, n_tok, H, seed=seed, device="cpu", commit=commit)
    d = to_device(x)
    return x, d


def contiguous_decode(d):
    S = d["S0"].clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], S, n_commit=d["n_commit"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, S


@pytest.mark.parametrize("n_tok,commit", [(1, "all"), (4, "random")])
def test_decode_paged_copy_equals_contiguous(n_tok, commit):
    """Read from scattered pages, write the committed state to other pages: the contiguous
    call's bits; the source pages stay unchanged (a shared snapshot may be speculated on)."""
    B, H = 6, 3
    x, d = decode_case(B, n_tok, H, seed=81 + n_tok, commit=commit)
    s_in, s_out = inputs.make_page_tables([B * H, B * H], 64, seed=81)
    pool = canary_pool(64, 7)
    pool[s_in.long()] = d["S0"].reshape(-1, 128, 128)
    before = pool.clone()
    o_ref, S_ref = contiguous_decode(d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.decode_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, s_in.cuda(), s_out.cuda(),
                         n_commit=d["n_commit"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o, o_ref)
    assert torch.equal(pool[s_out.long()], S_ref.reshape(-1, 128, 128))  # n_commit = 0: the entry state
    keep = torch.ones(64, dtype=torch.bool)
    keep[s_out.long()] = False
    assert torch.equal(pool[keep.cuda()], before[keep.cuda()])


def test_decode_paged_in_place_and_zero_entry():
    B, H = 4, 2
    x, d = decode_case(B, 4, H, seed=83, commit="random")
    s_in = torch.tensor([10, 3, -1, 7, 0, 12, 5, 9], dtype=torch.int32)
    pool = canary_pool(16, 8)
    S0 = torch.zeros(B * H, 128, 128, device="cuda")
    for u, pg in enumerate(s_in.tolist()):
        if pg >= 0:
            S0[u] = pool[pg]
    d["S0"] = S0.reshape(B, H, 128, 128)
    before = pool.clone()
    o_ref, S_ref = contiguous_decode(d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.decode_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, s_in.cuda(), None,
                         n_commit=d["n_commit"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(o, o_ref)
    flat = S_ref.reshape(-1, 128, 128)
    nc = x.n_commit.tolist()
    for u, pg in enumerate(s_in.tolist()):
        if pg >= 0:
            want = flat[u] if nc[u // H] > 0 else before[pg]
            assert torch.equal(pool[pg], want)


def test_decode_paged_against_the_oracle():
    B, H = 3, 2
    x, d = decode_case(B, 4, H, seed=84, commit="random")
    s_in, s_out = inputs.make_page_tables([B * H, B * H], 20, seed=84)
    pool = canary_pool(20, 9)
    pool[s_in.long()] = d["S0"].reshape(-1, 128, 128)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.decode_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, s_in.cuda(), s_out.cuda(),
                         n_commit=d["n_commit"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    import oracle
    from kda_gpu_util import bits
    ref = oracle.decode(bits(x.q), bits(x.k), bits(x.v), host(x.g), host(x.beta), host(x.S0),
                        x.n_commit.numpy().astype(np.int32))
    assert rel_max(host(o), ref["o"]) <= DECODE_TOL
    got = host(pool[s_out.long()]).reshape(B, H, 128, 128)
    assert rel_max(got, ref["S"]) <= DECODE_TOL


@pytest.mark.parametrize("bad", ["dup_out", "out_over_other_read", "in_place_dup", "out_of_pool"])
def test_decode_page_violations_write_nothing(bad):
    B, H = 2, 2
    x, d = decode_case(B, 1, H, seed=85, commit="all")
    s_in = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    s_out = torch.tensor([4, 5, 6, 7], dtype=torch.int32)
    if bad == "dup_out":
        s_out[2] = 4
    elif bad == "out_over_other_read":
        s_out[0] = 3
    elif bad == "in_place_dup":
        s_in[1] = 0
        s_out = None
    else:
        s_in[3] = 8
    pool = canary_pool(8, 10)
    before = pool.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = torch.full((B, 1, H, 128), float("nan"), device="cuda")
    kda.decode_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, s_in.cuda(),
                     None if s_out is None else s_out.cuda(), o=o, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == DEVICE_CHECK
    assert torch.isnan(o).all() and torch.equal(pool, before)


def test_decode_paged_mixed_tables():
    """Copy to fresh pages for some units, in place for others (out = in), -1 entries for a
    zero entry state and for no write, n_commit random: each unit as the contiguous call."""
    B, H = 4, 2
    x, d = decode_case(B, 4, H, seed=86, commit="random")
    s_in = torch.tensor([0, -1, 2, 3, 4, -1, 6, 7], dtype=torch.int32)
    s_out = torch.tensor([10, 11, 2, -1, 14, -1, 6, 17], dtype=torch.int32)
    pool = canary_pool(20, 11)
    S0 = torch.zeros(B * H, 128, 128, device="cuda")
    for u, pg in enumerate(s_in.tolist()):
        if pg >= 0:
            S0[u] = pool[pg]
    d["S0"] = S0.reshape(B, H, 128, 128)
    before = pool.clone()
    o_ref, S_ref = contiguous_decode(d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.decode_paged(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, s_in.cuda(), s_out.cuda(),
                         n_commit=d["n_commit"], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and torch.equal(o, o_ref)
    flat = S_ref.reshape(-1, 128, 128)
    nc = x.n_commit.tolist()
    written = set()
    for u, (pi, po) in enumerate(zip(s_in.tolist(), s_out.tolist())):
        if po < 0:
            continue
        written.add(po)
        if po == pi and nc[u // H] == 0:
            assert torch.equal(pool[po], before[po])  # in place, nothing committed: untouched
        else:
            assert torch.equal(pool[po], flat[u])     # a fresh page always takes the committed state
    keep = [p for p in range(20) if p not in written]
    assert torch.equal(pool[keep], before[keep])
