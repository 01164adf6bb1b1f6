"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics, not by the
oracle's own formula.  Each function raises AssertionError when the oracle disagrees.

Sources:
  [p1] "Kimi K3.1 Pro 架构完全拆解": 3.1 recurrence, 3.2 bounded log-decay, 3.4 replay
  [p2] "Kimi K3 的架構 ..." (SemiAnalysis translation): 4 delta rule, 6 FlashKDA algorithm
  [p3] "部署 Kimi K3 ...": 2 segment algebra, 3.3 restart at 2560 = 5 x 512
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle import chunked, segments


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def rand_case(T, H, d, seed, decay="sigmoid", s0_std=0.3, beta=None, g=None):
    rng = np.random.default_rng(seed)
    def unit(x):
        return x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = unit(rng.standard_normal((T, H, d))).astype(np.float32)
    k = unit(rng.standard_normal((T, H, d))).astype(np.float32)
    v = rng.standard_normal((T, H, d)).astype(np.float32)
    if beta is None:
        beta = sigmoid(rng.standard_normal((T, H))).astype(np.float32)
    else:
        beta = np.full((T, H), beta, np.float32)
    if g is None:
        if decay == "sigmoid":
            g = (-5.0 * sigmoid(rng.standard_normal((T, H, d)) - 4.0)).astype(np.float32)
        else:
            g = (-5.0 * (1.0 - rng.random((T, H, d)))).astype(np.float32)
    else:
        g = np.full((T, H, d), g, np.float32)
    S0 = None if s0_std is None else (rng.standard_normal((1, H, d, d)) * s0_std).astype(np.float32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, S0=S0)


def run(c, cu=None, every=False, **kw):
    T = c["q"].shape[0]
    cu = np.array([0, T], np.int32) if cu is None else np.asarray(cu, np.int32)
    off = pos = None
    if every:  # a checkpoint after every token: exposes S_t for all t
        lens = np.diff(cu)
        off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        pos = np.concatenate([np.arange(1, n + 1) for n in lens]).astype(np.int32)
    return oracle.prefill(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, S_in=c["S0"],
                          ckpt_off=off, ckpt_pos=pos, **kw)


def exact_unit_keys(n, d, seed):
    """Keys with entries +-1/4 on 16 channels: unit norm exactly in binary floating point."""
    rng = np.random.default_rng(seed)
    k = np.zeros((n, d), np.float32)
    for i in range(n):
        ch = rng.choice(d, 16, replace=False)
        k[i, ch] = rng.choice([-0.25, 0.25], 16)
    return k


def hadamard16():
    h = np.array([[1.0]])
    for _ in range(4):
        h = np.block([[h, h], [h, -h]])
    return h


# ---------------------------------------------------------------- closed forms [p1 3.1]
def pin_single_token():
    """From S = 0 one token gives S_1 = beta k v^T and o_1 = beta (q . k) v."""
    c = rand_case(1, 3, 32, seed=11, s0_std=None)
    r = run(c)
    for h in range(3):
        q, k, v = (c[x][0, h].astype(np.float64) for x in ("q", "k", "v"))
        b = float(c["beta"][0, h])
        np.testing.assert_allclose(r["S_out"][0, h], b * np.outer(k, v), rtol=0, atol=1e-14)
        np.testing.assert_allclose(r["o"][0, h], b * np.dot(q, k) * v, rtol=0, atol=1e-14)


def pin_decay_only():
    """beta = 0: S_t = Diag(exp(sum_{r<=t} g_r)) S_0 (natural exp), o_t = S_t^T q_t."""
    c = rand_case(40, 2, 24, seed=12, decay="uniform", beta=0.0)
    r = run(c, every=True)
    G = np.cumsum(c["g"].astype(np.float64), axis=0)
    for h in range(2):
        S0 = c["S0"][0, h].astype(np.float64)
        for t in (0, 7, 39):
            St = np.exp(G[t, h])[:, None] * S0
            np.testing.assert_allclose(r["ckpts"][t, h], St, rtol=1e-12, atol=1e-300)
            np.testing.assert_allclose(r["o"][t, h], St.T @ c["q"][t, h].astype(np.float64),
                                       rtol=1e-11, atol=1e-300)


def pin_identity_token():
    """beta = 0 and g = 0 leave the state bit-for-bit unchanged and o_t = S_0^T q_t."""
    c = rand_case(17, 2, 16, seed=13, beta=0.0, g=0.0)
    r = run(c)
    assert np.array_equal(r["S_out"][0], c["S0"][0].astype(np.float64))
    for h in range(2):
        np.testing.assert_allclose(r["o"][:, h], c["q"][:, h].astype(np.float64) @ c["S0"][0, h].astype(np.float64),
                                   rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------ delta rule [p2 4, p1 3.1]
def pin_retrieval():
    """beta = 1, |k| = 1: S_t^T k_t = v_t after every token, whatever the decay and S_0
    (the update overwrites the value stored under the current key; decay acts first)."""
    T, H, d = 30, 2, 64
    c = rand_case(T, H, d, seed=14, decay="uniform", beta=1.0)
    for h in range(H):
        c["k"][:, h] = exact_unit_keys(T, d, seed=100 + h)
    r = run(c, every=True)
    for t in range(T):
        for h in range(H):
            got = r["ckpts"][t, h].T @ c["k"][t, h].astype(np.float64)
            np.testing.assert_allclose(got, c["v"][t, h], rtol=0, atol=1e-12)


def pin_orthonormal_write():
    """alpha = 1, beta = 1, S_0 = 0, d orthonormal keys: afterwards S^T k_i = v_i for all i."""
    d = 64
    K = np.zeros((d, d))
    for b in range(d // 16):
        K[16 * b:16 * b + 16, 16 * b:16 * b + 16] = hadamard16() / 4.0
    perm = np.random.default_rng(15).permutation(d)
    K = K[perm]
    c = rand_case(d, 1, d, seed=15, beta=1.0, g=0.0, s0_std=None)
    c["k"][:, 0] = K.astype(np.float32)
    r = run(c)
    S = r["S_out"][0, 0]
    np.testing.assert_allclose(K @ S, c["v"][:, 0], rtol=0, atol=1e-13)


def pin_matrix_form():
    """Brute force on tiny d: S_t = (I - beta k k^T) Diag(exp g) S_{t-1} + beta k v^T with
    explicit d x d matrices, o_t = S_t^T q_t."""
    for d, seed in ((4, 16), (7, 17)):
        c = rand_case(12, 2, d, seed=seed, decay="uniform")
        r = run(c, every=True)
        for h in range(2):
            S = c["S0"][0, h].astype(np.float64)
            for t in range(12):
                k = c["k"][t, h].astype(np.float64)
                b = float(c["beta"][t, h])
                A = np.eye(d) - b * np.outer(k, k)
                S = A @ np.diag(np.exp(c["g"][t, h].astype(np.float64))) @ S + b * np.outer(k, c["v"][t, h])
                np.testing.assert_allclose(r["ckpts"][t, h], S, rtol=1e-12, atol=1e-14)
                np.testing.assert_allclose(r["o"][t, h], S.T @ c["q"][t, h], rtol=1e-12, atol=1e-14)


def pin_linearity():
    """For fixed q, k, g, beta the result is linear in (S_0, V) jointly."""
    c = rand_case(50, 2, 32, seed=18, decay="uniform")
    full = run(c)
    c_s = dict(c, v=np.zeros_like(c["v"]))
    c_v = dict(c, S0=None)
    a, b = run(c_s), run(c_v)
    np.testing.assert_allclose(full["S_out"], a["S_out"] + b["S_out"], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(full["o"], a["o"] + b["o"], rtol=1e-11, atol=1e-13)


# ------------------------------------------------------- chunk form [p2 6] and [p1 3.2]
def pin_chunk_form(Cs=(1, 2, 4, 16, 64), Ts=(1, 5, 63, 64, 65, 130, 300)):
    """The chunk-level matrix form equals the per-token oracle (partial last chunks
    included), for both the typical and the stress decay distribution."""
    for decay, seed in (("sigmoid", 19), ("uniform", 20)):
        c = rand_case(max(Ts), 1, 32, seed=seed, decay=decay)
        for T in Ts:
            cc = {k: (v[:T] if k != "S0" else v) for k, v in c.items()}
            ref = run(cc)
            for C in Cs:
                O, S = chunked.prefill_one(cc["q"][:, 0], cc["k"][:, 0], cc["v"][:, 0], cc["g"][:, 0],
                                           cc["beta"][:, 0], cc["S0"][0, 0], C)
                scale = np.abs(ref["o"]).max()
                np.testing.assert_allclose(O, ref["o"][:, 0], rtol=0, atol=1e-9 * scale)
                np.testing.assert_allclose(S, ref["S_out"][0, 0], rtol=0, atol=1e-9 * np.abs(S).max())


# ------------------------------------------------------------- segment algebra [p3 2]
def pin_segments():
    """Exit state = S~ + M S_in for a split anywhere; the combine is associative; M is the
    state reached from S_in = I with V = 0."""
    T, d = 90, 16
    c = rand_case(T, 1, d, seed=21, decay="uniform")
    ref = run(c)
    S_in = c["S0"][0, 0].astype(np.float64)

    def pair(a, b):
        sub = {k: (v[a:b] if k != "S0" else None) for k, v in c.items()}
        St = run(sub)["S_out"][0, 0]
        return segments.transition(c["k"][a:b, 0], c["g"][a:b, 0], c["beta"][a:b, 0]), St

    for cuts in ((0, 37, T), (0, 1, 50, T), (0, 30, 60, T)):
        pairs = [pair(a, b) for a, b in zip(cuts[:-1], cuts[1:])]
        _, S_exit = segments.entry_states(pairs, S_in)
        np.testing.assert_allclose(S_exit, ref["S_out"][0, 0], rtol=0, atol=1e-11)
    p1, p2, p3 = pair(0, 20), pair(20, 55), pair(55, T)
    L = segments.combine(segments.combine(p1, p2), p3)
    R = segments.combine(p1, segments.combine(p2, p3))
    np.testing.assert_allclose(L[0], R[0], atol=1e-12)
    np.testing.assert_allclose(L[1], R[1], atol=1e-12)
    cI = dict(c, v=np.zeros_like(c["v"]), S0=np.eye(d, dtype=np.float32)[None, None])
    np.testing.assert_allclose(run(cI)["S_out"][0, 0],
                               segments.transition(c["k"][:, 0], c["g"][:, 0], c["beta"][:, 0]),
                               rtol=0, atol=1e-12)


# ------------------------------------------- packing, checkpoints, restart [p3 3.2-3.3]
def pin_restart_2560():
    """A request matched up to 2800 tokens resumes at 2560 = 5 x 512: resuming from the
    checkpoint at 2560 with the remaining tokens reproduces the continuous run."""
    T, H, d, P = 2800, 2, 16, 2560
    c = rand_case(T, H, d, seed=22)
    off = np.array([0, T // 512], np.int32)
    pos = np.arange(512, T + 1, 512, dtype=np.int32)
    full = oracle.prefill(c["q"], c["k"], c["v"], c["g"], c["beta"], np.array([0, T], np.int32),
                          S_in=c["S0"], ckpt_off=off, ckpt_pos=pos)
    assert list(pos) == [512, 1024, 1536, 2048, 2560]
    ck = full["ckpts"][list(pos).index(P)]
    tail = {k: (v[P:] if k != "S0" else ck[None].astype(np.float32)) for k, v in c.items()}
    rest = run(tail)
    np.testing.assert_allclose(rest["S_out"][0], full["S_out"][0], rtol=0, atol=1e-6)
    np.testing.assert_allclose(rest["o"], full["o"][P:], rtol=0, atol=1e-6)


def pin_packing_and_checkpoints():
    """Packed sequences equal separate runs bit for bit; the checkpoint at p = len is
    S_out; the checkpoint at p equals the final state of the run truncated to p tokens;
    unit and row subsets reproduce the full run."""
    lens = [5, 64, 1, 100, 33]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T, H, d = int(cu[-1]), 3, 16
    c = rand_case(T, H, d, seed=23, decay="uniform")
    rng = np.random.default_rng(23)
    c["S0"] = (rng.standard_normal((len(lens), H, d, d)) * 0.1).astype(np.float32)
    pos, off = [], [0]
    for n in lens:
        p = sorted(set(rng.choice(np.arange(1, n + 1), size=min(3, n), replace=False).tolist()) | {n})
        pos += p
        off.append(len(pos))
    off, pos = np.array(off, np.int32), np.array(pos, np.int32)
    full = oracle.prefill(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, S_in=c["S0"],
                          ckpt_off=off, ckpt_pos=pos)
    for i, n in enumerate(lens):
        a, b = cu[i], cu[i + 1]
        sub = {k: (v[a:b] if k != "S0" else v[i:i + 1]) for k, v in c.items()}
        one = run(sub)
        assert np.array_equal(one["o"], full["o"][a:b])
        assert np.array_equal(one["S_out"][0], full["S_out"][i])
        for j in range(off[i], off[i + 1]):
            p = int(pos[j])
            trunc = run({k: (v[:p] if k != "S0" else v) for k, v in sub.items()})
            assert np.array_equal(trunc["S_out"][0], full["ckpts"][j])
        assert np.array_equal(full["ckpts"][off[i + 1] - 1], full["S_out"][i])
    units = np.array([1, 5, 14], np.int64)
    rows = np.array([0, 3, 70, T - 1], np.int64)
    part = oracle.prefill(c["q"], c["k"], c["v"], c["g"], c["beta"], cu, S_in=c["S0"],
                          units=units, o_rows=rows)
    for u in units:
        s, h = divmod(int(u), H)
        assert np.array_equal(part["S_out"][s, h], full["S_out"][s, h])
        for ri, r in enumerate(rows):
            if cu[s] <= r < cu[s + 1]:
                assert np.array_equal(part["o"][ri, h], full["o"][r, h])


def pin_decode_commit():
    """Verify step [p1 3.4, p3 4]: outputs of all n_tok tokens, state after n_commit."""
    B, n, H, d = 5, 4, 2, 16
    c = rand_case(B * n, H, d, seed=24)
    rng = np.random.default_rng(24)
    S0 = (rng.standard_normal((B, H, d, d)) * 0.02).astype(np.float32)
    n_commit = np.array([0, 1, 2, 3, 4], np.int32)
    shp = lambda x: x.reshape((B, n) + x.shape[1:])
    r = oracle.decode(shp(c["q"]), shp(c["k"]), shp(c["v"]), shp(c["g"]), shp(c["beta"]), S0, n_commit)
    for b in range(B):
        sub = {k: v[b * n:(b + 1) * n] for k, v in c.items() if k != "S0"}
        sub["S0"] = S0[b:b + 1]
        ref = run(sub, every=True)
        assert np.array_equal(r["o"][b], ref["o"])
        want = S0[b].astype(np.float64) if n_commit[b] == 0 else ref["ckpts"][n_commit[b] - 1]
        assert np.array_equal(r["S"][b], want)


ALL_PINS = [pin_single_token, pin_decay_only, pin_identity_token, pin_retrieval,
            pin_orthonormal_write, pin_matrix_form, pin_linearity, pin_chunk_form,
            pin_segments, pin_restart_2560, pin_packing_and_checkpoints, pin_decode_commit]


# ------------------------------------------------------------------ output epilogue
# "Kimi K3.1 Pro 架构完全拆解" section 3.3: y = W_o [Sigmoid(W_g x) (.) RMSNorm(o~)], the
# bracket computed by oracle.epilogue.gated_rmsnorm.
def pin_epilogue_hand_values():
    """d = 4, o = (1, -2, 2, -4): mean square 25/4, so with eps = 0 the norm is o / 2.5;
    gate logits (0, 0, ln 3, -ln 3) give sigmoids (1/2, 1/2, 3/4, 1/4); gamma = (1, 2, 1, 4)."""
    from oracle.epilogue import gated_rmsnorm
    o = np.array([1.0, -2.0, 2.0, -4.0])
    a = np.array([0.0, 0.0, np.log(3.0), -np.log(3.0)])
    gam = np.array([1.0, 2.0, 1.0, 4.0])
    want = np.array([0.5 * 1 * 1 / 2.5, 0.5 * 2 * -2 / 2.5, 0.75 * 1 * 2 / 2.5, 0.25 * 4 * -4 / 2.5])
    got = gated_rmsnorm(o, a, gam, eps=0.0)
    assert np.allclose(got, want, rtol=1e-15, atol=0), (got, want)


def pin_epilogue_invariants():
    """With eps = 0: scale invariance z(c o) = z(o) for c > 0, sign flip z(-o) = -z(o), unit
    root-mean-square of the normalised row (gate logits -> +inf, gamma = 1), and a sigmoid of
    0 halves it; eps > 0 shrinks rows with a small norm (o = 0 maps to 0)."""
    from oracle.epilogue import gated_rmsnorm, sigmoid
    rng = np.random.default_rng(5)
    o = rng.standard_normal((3, 128))
    a = rng.standard_normal((3, 128))
    z = gated_rmsnorm(o, a, eps=0.0)
    assert np.allclose(gated_rmsnorm(7.5 * o, a, eps=0.0), z, rtol=1e-13)
    assert np.allclose(gated_rmsnorm(-o, a, eps=0.0), -z, rtol=1e-13)
    big = np.full_like(o, 60.0)
    n = gated_rmsnorm(o, big, eps=0.0)
    assert np.allclose(np.sqrt(np.mean(n * n, axis=-1)), 1.0, rtol=1e-13)
    h = gated_rmsnorm(o, np.zeros_like(o), eps=0.0)
    assert np.allclose(h, 0.5 * n, rtol=1e-13)
    assert np.all(gated_rmsnorm(np.zeros((2, 8)), np.zeros((2, 8)), eps=1e-5) == 0.0)
    s = 1e-3 * o
    shr = gated_rmsnorm(s, big, eps=1e-5)
    assert np.all(np.sqrt(np.mean(shr * shr, axis=-1)) < 1.0)
    assert np.allclose(sigmoid(np.array([-800.0, 0.0, 800.0])), [0.0, 0.5, 1.0], atol=0)


def pin_epilogue_eps_closed_form():
    """A constant row o = c (mean square c^2) with eps > 0 normalises to c / sqrt(c^2 + eps):
    c = 0.01, eps = 1e-4 gives 1 / sqrt(2) (times sigmoid and gamma)."""
    from oracle.epilogue import gated_rmsnorm
    o = np.full(128, 0.01)
    z = gated_rmsnorm(o, np.zeros(128), np.full(128, 2.0), eps=1e-4)
    assert np.allclose(z, 0.5 * 2.0 / np.sqrt(2.0), rtol=1e-14), z[:4]


ALL_PINS += [pin_epilogue_hand_values, pin_epilogue_invariants, pin_epilogue_eps_closed_form]


def pin_value_rotation():
    """The recurrence acts on the value side (d_v) by right multiplication only
    ([p1] 3.1: S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T): for any orthogonal R,
    v -> v R and S0 -> S0 R give o -> o R and S -> S R.  A transposed state or read-out, or a
    decay applied on the value side, breaks it."""
    T, H, d = 37, 2, 16
    c = rand_case(T, H, d, seed=41)
    rng = np.random.default_rng(42)
    R, _ = np.linalg.qr(rng.standard_normal((d, d)))
    base = run(c)
    c2 = dict(c)
    c2["v"] = (c["v"].astype(np.float64) @ R).astype(np.float32)
    c2["S0"] = (c["S0"].astype(np.float64) @ R).astype(np.float32)
    rot = run(c2)
    want_o = base["o"] @ R
    want_S = base["S_out"] @ R
    scale = np.abs(want_o).max()
    assert np.abs(rot["o"] - want_o).max() <= 1e-5 * scale, np.abs(rot["o"] - want_o).max()
    assert np.abs(rot["S_out"] - want_S).max() <= 1e-5 * np.abs(want_S).max()


def pin_key_permutation():
    """The decay is diagonal in d_k ([p1] 3.1-3.2): permuting the key channels of q, k, g
    and the rows of S0 together leaves o unchanged and permutes the rows of S.  A decay
    applied on the wrong axis or a mixed-up channel index breaks it."""
    T, H, d = 29, 2, 16
    c = rand_case(T, H, d, seed=43, decay="uniform")
    perm = np.random.default_rng(44).permutation(d)
    base = run(c)
    c2 = dict(c)
    for key in ("q", "k", "g"):
        c2[key] = np.ascontiguousarray(c[key][..., perm])
    c2["S0"] = np.ascontiguousarray(c["S0"][:, :, perm, :])
    pm = run(c2)
    assert np.allclose(pm["o"], base["o"], rtol=1e-12, atol=1e-14)
    assert np.allclose(pm["S_out"], base["S_out"][:, :, perm, :], rtol=1e-12, atol=1e-14)


ALL_PINS += [pin_value_rotation, pin_key_permutation]


# --------------------------------------------------------------------- decode front end
# oracle/frontend.py: "Kimi K3 的架構 ... 服務性能" section 7 (short causal convolution, q/k L2
# normalisation, alpha and beta gates) and "Kimi K3.1 Pro 架构完全拆解" 3.2 (bounded decay
# gate) and 3.4 (fused replay step).

def pin_frontend_conv_against_numpy():
    """Each channel of the causal convolution equals numpy.convolve of (cache, x) with the
    channel's filter, taken at the positions of the n tokens; W = 1 with tap 1 is the
    identity; an input never changes an earlier output."""
    from oracle.frontend import short_conv
    rng = np.random.default_rng(11)
    for W in (1, 2, 3, 4):
        x = rng.standard_normal((6, 5))
        cache = rng.standard_normal((W - 1, 5))
        w = rng.standard_normal((5, W))
        y = short_conv(x, cache, w)
        full = np.concatenate([cache, x], 0)
        for c in range(5):
            want = np.convolve(full[:, c], w[c])[W - 1:W - 1 + 6]
            assert np.allclose(y[:, c], want, rtol=1e-13, atol=1e-13), (W, c)
        x2 = x.copy()
        x2[3] += 10.0
        assert np.array_equal(short_conv(x2, cache, w)[:3], y[:3])
    x = rng.standard_normal((4, 3))
    assert np.array_equal(short_conv(x, np.zeros((0, 3)), np.ones((3, 1))), x)


def pin_frontend_silu_and_l2():
    """SiLU: silu(0) = 0, silu(1) = 1 / (1 + e^-1), silu(x) -> x for large x and -> 0 for very
    negative x.  L2: (3, 4) -> (0.6, 0.8), unit norm, scale invariance, zero stays zero."""
    from oracle.frontend import l2_normalize, short_conv, silu
    assert silu(0.0) == 0.0
    assert np.isclose(silu(1.0), 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)
    assert np.isclose(silu(40.0), 40.0, rtol=1e-15) and abs(silu(-40.0)) < 1e-15
    x = np.array([[0.5, -1.0]])
    y = short_conv(x, np.zeros((0, 2)), np.ones((2, 1)), act="silu")
    assert np.allclose(y, [[0.5 / (1 + np.exp(-0.5)), -1.0 / (1 + np.exp(1.0))]], rtol=1e-15)
    assert np.allclose(l2_normalize(np.array([3.0, 4.0])), [0.6, 0.8], rtol=1e-15)
    rng = np.random.default_rng(12)
    v = rng.standard_normal((4, 128))
    u = l2_normalize(v)
    assert np.allclose(np.linalg.norm(u, axis=-1), 1.0, rtol=1e-14)
    assert np.allclose(l2_normalize(3.7 * v), u, rtol=1e-14)
    assert np.array_equal(l2_normalize(np.zeros((2, 8))), np.zeros((2, 8)))


def pin_frontend_gates():
    """g = g_min Sigmoid(e^A z): z = 0 gives g_min / 2; z = ln 3, A = 0 gives Sigmoid = 3/4,
    g = -3.75 at g_min = -5; A rescales z (g(z, A) = g(z e^A, 0)); g stays in (g_min, 0) and
    alpha = e^g >= e^g_min.  beta = Sigmoid(b): 1/2 at 0, 3/4 at ln 3, b -> -b gives 1 - beta."""
    from oracle.frontend import beta_gate, decay_log
    assert decay_log(0.0, 0.3) == -2.5
    assert np.isclose(decay_log(np.log(3.0), 0.0), -3.75, rtol=1e-15)
    assert np.isclose(decay_log(np.log(3.0), 0.0, g_min=-2.0), -1.5, rtol=1e-15)
    rng = np.random.default_rng(13)
    z = rng.standard_normal(1000) * 3
    a = rng.standard_normal(1000)
    assert np.allclose(decay_log(z, a), decay_log(z * np.exp(a), 0.0), rtol=1e-14)
    g = decay_log(z, a)
    assert np.all(g <= 0) and np.all(g >= -5.0) and np.all(np.exp(g) >= np.exp(-5.0))
    mid = np.abs(z * np.exp(a)) < 30  # away from the sigmoid's fp64 saturation the bounds are strict
    assert np.all(g[mid] < 0) and np.all(g[mid] > -5.0)
    assert beta_gate(0.0) == 0.5 and np.isclose(beta_gate(np.log(3.0)), 0.75, rtol=1e-15)
    assert np.allclose(beta_gate(-z), 1.0 - beta_gate(z), rtol=1e-13, atol=1e-15)


def _frontend_case(rng, B=2, n=4, H=2, d=16, W=4):
    qp, kp, vp = (rng.standard_normal((B, n, H, d)) for _ in range(3))
    conv_w = rng.standard_normal((3, H, d, W)) * 0.5
    cache = rng.standard_normal((B, H, 3, W - 1, d))
    z = rng.standard_normal((B, n, H, d)) - 2.0
    a_log = rng.standard_normal(H) * 0.3
    b = rng.standard_normal((B, n, H))
    S = rng.standard_normal((B, H, d, d)) * 0.1
    return qp, kp, vp, conv_w, cache, z, a_log, b, S


def pin_frontend_replay_identities():
    """A step over tokens 0..1 followed by a step over tokens 2..4 (from the state and cache
    the first left) gives the outputs and final state of one step over tokens 0..4; a step
    that commits only its first m tokens leaves the state and cache of a step over those m
    tokens alone; n_commit = 0 leaves both unchanged."""
    from oracle.frontend import decode_step
    rng = np.random.default_rng(14)
    qp, kp, vp, conv_w, cache, z, a_log, b, S = _frontend_case(rng, n=5)
    for act in ("none", "silu"):
        one = decode_step(qp, kp, vp, conv_w, cache, z, a_log, b, S, act=act)
        sl = lambda t, a, e: t[:, a:e]
        r1 = decode_step(sl(qp, 0, 2), sl(kp, 0, 2), sl(vp, 0, 2), conv_w, cache, sl(z, 0, 2), a_log, sl(b, 0, 2), S,
                         act=act)
        r2 = decode_step(sl(qp, 2, 5), sl(kp, 2, 5), sl(vp, 2, 5), conv_w, r1["conv_cache"], sl(z, 2, 5), a_log,
                         sl(b, 2, 5), r1["S"], act=act)
        assert np.allclose(np.concatenate([r1["o"], r2["o"]], 1), one["o"], rtol=1e-11, atol=1e-12)
        assert np.allclose(r2["S"], one["S"], rtol=1e-11, atol=1e-12)
        assert np.allclose(r2["conv_cache"], one["conv_cache"], rtol=0, atol=0)
    part = decode_step(qp[:, :4], kp[:, :4], vp[:, :4], conv_w, cache, z[:, :4], a_log, b[:, :4], S,
                       n_commit=np.array([2, 0]))
    two = decode_step(qp[:, :2], kp[:, :2], vp[:, :2], conv_w, cache, z[:, :2], a_log, b[:, :2], S)
    assert np.allclose(part["S"][0], two["S"][0], rtol=1e-13, atol=1e-15)
    assert np.array_equal(part["conv_cache"][0], two["conv_cache"][0])
    assert np.array_equal(part["S"][1], S[1]) and np.array_equal(part["conv_cache"][1], cache[1])
    assert np.allclose(part["o"][:, :2], two["o"], rtol=1e-13, atol=1e-15)  # outputs never depend on n_commit


def pin_frontend_recurrence_against_c_oracle():
    """The batched numpy recurrence equals the C oracle's decode (an independent
    implementation of the same definition) on the same fp32-representable inputs."""
    import oracle
    from oracle.frontend import l2_normalize, recurrence
    rng = np.random.default_rng(15)
    B, n, H, d = 3, 4, 2, 128
    f32 = lambda t: np.asarray(t, np.float32)
    q = f32(l2_normalize(rng.standard_normal((B, n, H, d))))
    k = f32(l2_normalize(rng.standard_normal((B, n, H, d))))
    v = f32(rng.standard_normal((B, n, H, d)))
    g = f32(-5.0 / (1.0 + np.exp(-(rng.standard_normal((B, n, H, d)) - 2.0))))
    beta = f32(1.0 / (1.0 + np.exp(-rng.standard_normal((B, n, H)))))
    S = f32(rng.standard_normal((B, H, d, d)) * 0.05)
    nc = np.array([4, 1, 0], np.int32)
    o, Sn = recurrence(q, k, v, g, beta, S, nc)
    ref = oracle.decode(q, k, v, g, beta, S, nc)
    assert np.allclose(o, ref["o"], rtol=1e-10, atol=1e-12)
    assert np.allclose(Sn, ref["S"], rtol=1e-10, atol=1e-12)


def pin_frontend_step_retrieval():
    """The fused step's key reaches the recurrence unit-normalised: with beta = 1 (b large)
    the delta rule makes the new state return the token's value, S_new^T k = v, exactly when
    ||k|| = 1 ("Kimi K3 ... 服務性能" 4 and 7); the value is the convolution's output (identity
    filter of width 1: v = vp) and the query and key have unit norm."""
    from oracle.frontend import decode_step
    rng = np.random.default_rng(16)
    B, H, d = 2, 2, 32
    qp, kp, vp = (rng.standard_normal((B, 1, H, d)) * 3 for _ in range(3))
    ones = np.ones((3, H, d, 1))
    z = rng.standard_normal((B, 1, H, d))
    b = np.full((B, 1, H), 60.0)
    S = rng.standard_normal((B, H, d, d))
    r = decode_step(qp, kp, vp, ones, np.zeros((B, H, 3, 0, d)), z, np.zeros(H), b, S)
    assert np.allclose(np.linalg.norm(r["k"], axis=-1), 1.0, rtol=1e-14)
    assert np.allclose(np.linalg.norm(r["q"], axis=-1), 1.0, rtol=1e-14)
    assert np.array_equal(r["v"], vp)
    k, v = r["k"][:, 0], r["v"][:, 0]
    assert np.allclose(np.einsum("bhij,bhi->bhj", r["S"], k), v, rtol=1e-12, atol=1e-12)


ALL_PINS += [pin_frontend_conv_against_numpy, pin_frontend_silu_and_l2, pin_frontend_gates,
             pin_frontend_replay_identities, pin_frontend_recurrence_against_c_oracle,
             pin_frontend_step_retrieval]
