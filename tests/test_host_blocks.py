"""Block planning of kda_prefill_host (host only, no GPU): the borders cover the packed
stream in order, each border that cuts a sequence sits on that sequence's chunk grid (a
multiple of 64 tokens from its start, so the blocks go through the chunks of one call),
blocks stay near the requested size, and bad inputs are refused."""
import random

import pytest
import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return kda.library()


def cu_of(lengths):
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + n)
    return torch.tensor(cu, dtype=torch.int32)


def check_borders(lengths, block):
    cu = cu_of(lengths)
    b = kda.prefill_host_blocks(cu, block)
    T = int(cu[-1])
    if not lengths:
        return b
    assert b[0] == 0 and b[-1] == T
    if T == 0:
        assert b == [0, 0]
        return b
    assert all(x < y for x, y in zip(b, b[1:])), b
    target = block or max(1024, (T // 8 + 63) // 64 * 64)
    c = cu.tolist()
    for x in b[1:-1]:
        inside = [s for s in range(len(lengths)) if c[s] < x < c[s + 1]]
        if inside:
            assert (x - c[inside[0]]) % 64 == 0, (x, c[inside[0]])
    for x, y in zip(b, b[1:]):
        assert y - x <= target + 63
    return b


def test_hand_example():
    """cu = (0, 5, 69, 70, 200, 200, 277) with 64-token blocks: 5 (a border inside
    sequence 1 would be off its grid), 69, 70, then sequence 3 on its grid (134, 198),
    200, 264, 277."""
    assert check_borders([5, 64, 1, 130, 0, 77], 64) == [0, 5, 69, 70, 134, 198, 200, 264, 277]


def test_single_sequence_default():
    """1024-token blocks; the final stretch (1024 tokens) ends with a 256-token block, the
    part of the pipeline no upload overlaps."""
    assert check_borders([8192], 0) == list(range(0, 8192, 1024)) + [7936, 8192]
    assert check_borders([100], 0) == [0, 100]
    assert check_borders([600], 0) == [0, 320, 600]  # tail split at 344, moved down to the chunk grid
    assert check_borders([500], 0) == [0, 500]        # at most 2 x 256 tokens: one block


@pytest.mark.parametrize("seed", range(20))
def test_random_packings(seed):
    rng = random.Random(seed)
    lengths = [rng.choice([0, 1, 63, 64, 65, rng.randint(1, 3000)]) for _ in range(rng.randint(1, 12))]
    block = rng.choice([64, 128, 512, 1024, 0])
    T = sum(lengths)
    if T and (T + block - 1) // max(block, 1) > 60 and block:
        block = 64 * ((T // 50) // 64 + 1)
    check_borders(lengths, block)


def test_refusals():
    with pytest.raises(ValueError):
        kda.prefill_host_blocks(cu_of([100]), 100)  # not a multiple of 64
    with pytest.raises(ValueError):
        kda.prefill_host_blocks(cu_of([64 * 65]), 64)  # 65 blocks
    with pytest.raises(ValueError):
        kda.prefill_host_blocks(torch.tensor([0, 10, 5], dtype=torch.int32), 64)  # decreasing offsets
    assert kda.prefill_host_blocks(cu_of([0, 0]), 64) == [0, 0]
