"""The output stage's bar (``kda_gpu_util.y_bound``) on the CPU: it admits every y that an o~
within the o bar produces once y is rounded to bf16, and it rejects the plausible mistakes
in the stage ("Kimi K3.1 Pro 架构完全拆解" 3.3: y = sigmoid(a) (.) RMSNorm(o~), with weight
w and eps inside the root).  No GPU."""
import numpy as np
import torch

from kda_gpu_util import O_TOL, y_bound
from oracle.epilogue import gated_rmsnorm, sigmoid

EPS = 1e-5


def _rows(seed, n=256, d=128):
    rng = np.random.default_rng(seed)
    scale = np.exp(rng.uniform(np.log(1e-3), 0.0, size=(n, 1)))  # rows from 1e-3 to 1 of the max
    o = rng.standard_normal((n, d)) * scale
    a = rng.standard_normal((n, d)) * 2.0
    w = 1.0 + 0.1 * rng.standard_normal(d)
    return o, a, w


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


def _ratio(y, o, a, w, eps=EPS):
    bound, yr = y_bound(o, a, w, eps, np.abs(o).max())
    return float((np.abs(y - yr) / bound).max())


def test_bar_admits_o_within_its_bar():
    for seed in range(6):
        o, a, w = _rows(seed)
        eps_o = O_TOL * np.abs(o).max()
        rng = np.random.default_rng(100 + seed)
        # worst-shaped perturbations of the full allowed size: all +eps_o, alternating
        # signs, and random signs; each then rounded to bf16 like the kernel's output
        for delta in (np.full_like(o, eps_o), eps_o * np.where(np.arange(o.shape[1]) % 2, 1.0, -1.0),
                      eps_o * rng.choice([-1.0, 1.0], size=o.shape), -eps_o * np.sign(o)):
            y = _bf16(gated_rmsnorm(o + delta, a, w, EPS))
            assert _ratio(y, o, a, w) <= 1.0


def test_bar_rejects_planted_mistakes():
    o, a, w = _rows(7)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    mistakes = {
        "gate_negated": sigmoid(-a) * w * o / np.sqrt(ms + EPS),
        "gate_missing": w * o / np.sqrt(ms + EPS),
        "gate_not_sigmoid": np.tanh(a) * w * o / np.sqrt(ms + EPS),
        "weight_dropped": sigmoid(a) * o / np.sqrt(ms + EPS),
        "sum_not_mean": sigmoid(a) * w * o / np.sqrt(128 * ms + EPS),
        "no_root": sigmoid(a) * w * o / (ms + EPS),
        "norm_over_all_rows": sigmoid(a) * w * o / np.sqrt(np.mean(o * o) + EPS),
    }
    for name, y in mistakes.items():
        assert _ratio(_bf16(y), o, a, w) > 1.0, name


def test_bar_rejects_eps_outside_the_root():
    # with a large eps the placement of eps matters; the bar must see it
    o, a, w = _rows(8)
    eps = 1e-2
    ms = np.mean(o * o, axis=-1, keepdims=True)
    y = sigmoid(a) * w * o / (np.sqrt(ms) + eps)
    assert _ratio(_bf16(y), o, a, w, eps) > 1.0
