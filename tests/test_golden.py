"""Printed figures from the pages, recomputed from their stated arithmetic."""
import math
import os

import torch

from kimi_delta_attention_prefill_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def _figures():
    out = {}
    for line in open(os.path.join(HERE, "golden", "printed_figures.txt"), encoding="utf-8"):
        line = line.split("#", 1)[0].strip()
        if line:
            key, rest = line.split("=", 1)
            out[key.strip()] = float(rest.split(";", 1)[0])
    return out


F = _figures()


def sig2(x):
    return float(f"{x:.2g}")


def test_decay_floor_and_range():
    assert inputs.G_MIN == F["g_min"]
    assert sig2(math.exp(F["g_min"])) == F["retention_floor"]
    assert 16 * F["g_min"] == F["tile16_logdecay_floor"]
    assert sig2(math.exp(-F["tile16_logdecay_floor"])) == F["rescale_bound"]
    bf16_max = torch.finfo(torch.bfloat16).max
    assert sig2(bf16_max) == F["bf16_max"]
    assert math.exp(-F["tile16_logdecay_floor"]) < bf16_max


def test_state_size():
    assert round(69 * 96 * 128 * 128 * 2 / 2**20) == F["state_mib_69_layers_96_heads"]


def test_analytic_counts():
    D, C = 128, 64
    assert 7 * D * D == F["decode_flops_per_head_token"]
    assert 8 * D * D == F["decode_bytes_per_head_token"]
    assert 12 * C**3 + 8 * C**2 * D + 6 * C * D**2 == F["prefill_flops_per_chunk_head"]


def test_restart_position():
    hb = int(F["hash_block"])
    assert (int(F["restart_match"]) // hb) * hb == F["restart_at"] == 5 * hb


def test_generator_decay_range():
    x = inputs.make_prefill([300], H=2, d=16, seed=0, decay="uniform")
    assert float(x.g.min()) >= F["g_min"] and float(x.g.max()) < 0
    y = inputs.make_prefill([300], H=2, d=16, seed=0, decay="sigmoid")
    assert float(y.g.min()) > F["g_min"] and float(y.g.max()) < 0
    n = torch.linalg.vector_norm(y.k.float(), dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-2)
