"""Cross-device sequence split (KCP) over torch.distributed: the exchange around the two
device parts ``kda_prefill_pairs`` / ``kda_combine_pairs`` and the ordinary prefill.

"部署 Kimi K3：从 KDA Kernel 到 Fleet 调度的推理 Infra 全景", section 2: a sequence too long
for one device is split over ranks in token order.  A rank's token range acts on the state
as the pair (M, S~) -- cumulative transition and zero-entry state -- whose size (2 x 64 KiB
per head) does not depend on the tokens.  Each rank computes its pair, the ranks exchange
them in one all-gather, each folds the pairs of the ranks before it onto the sequence's
entry state (a local sequential combine), and runs its own range from that true entry
state.  One call, on every rank of ``group``, in this order:

  1. device part: the pair (M, S~) of this rank's rows of every sequence;
  2. readiness (host): the rank posts "ok" with its shapes under the call's key in
     ``store`` and waits, with a time limit counted from its own post, for every other
     rank's post; a rank whose pair failed posts "failed" and leaves at once.  A failed or
     missing rank, or a shape mismatch, ends the call on every rank with
     :class:`KcpError` before any collective is entered;
  3. one all-gather of the pairs (NCCL on GPUs, gloo on the host);
  4. device part: the combine of ranks 0 .. rank-1's pairs onto the entry states;
  5. device part: this rank's rows from the true entry states.

Ranks pass the same sequences (``n_seq`` and ``H`` alike); a rank may hold no rows of a
sequence.  Every rank passes the sequences' entry states ``S_in`` (or None for zeros).
Everything a rank receives lands in its own memory first (all-gather into local tensors).
The device parts are pluggable (:class:`DeviceParts`): :func:`gpu_parts` runs them in the
library's kernels; the tests substitute the CPU oracle to check the exchange alone.
"""
from __future__ import annotations

import datetime
import itertools
from dataclasses import dataclass
from typing import Any, Callable

import torch

__all__ = ["KcpError", "DeviceParts", "gpu_parts", "kcp_prefill"]

_calls = itertools.count()


class KcpError(RuntimeError):
    """The call could not complete on every rank (a rank failed, was missing, or disagreed)."""


@dataclass
class DeviceParts:
    """The per-rank work of a call.  ``pairs(local) -> (M, S_tilde)`` with shapes
    ``[N, H, d, d]``; ``combine(M, S_tilde, S_in) -> entry`` with ``[R, N, H, d, d]`` pairs of
    the preceding ranks; ``run(local, entry) -> result`` (the rank's outputs)."""
    pairs: Callable[[Any], tuple]
    combine: Callable[[torch.Tensor, torch.Tensor, Any], torch.Tensor]
    run: Callable[[Any, torch.Tensor], Any]


def gpu_parts(**prefill_kwargs) -> DeviceParts:
    """Device parts in the library's kernels.  ``local`` is a mapping with the rank's rows:
    q, k, v, g, beta and cu_seqlens (CUDA tensors, as :func:`prefill`); extra keyword
    arguments go to :func:`prefill` in the last step (checkpoints, a workspace, ...)."""
    from . import combine_pairs, prefill, prefill_pairs

    def pairs(x):
        return prefill_pairs(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"])

    def combine(M, St, S_in):
        return combine_pairs(M.contiguous(), St.contiguous(), S_in=S_in)

    def run(x, entry):
        return prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], S_in=entry, **prefill_kwargs)

    return DeviceParts(pairs, combine, run)


def _post_and_wait(store, tag, rank, world, mine, timeout_s):
    store.set(f"{tag}/{rank}", mine)
    keys = [f"{tag}/{r}" for r in range(world)]
    try:
        store.wait(keys, datetime.timedelta(seconds=timeout_s))
    except Exception as e:  # the store reports a timeout with its own exception types
        missing = [r for r in range(world) if not store.check([f"{tag}/{r}"])]
        raise KcpError(f"rank(s) {missing} did not post within {timeout_s} s ({type(e).__name__})") from None
    return [store.get(k).decode() for k in keys]


def kcp_prefill(local, S_in, store, group=None, parts: DeviceParts | None = None, timeout_s: float = 30.0,
                tag: str | None = None):
    """One cross-device prefill call on this rank (see the module docstring).

    ``local``: this rank's rows (passed to ``parts``); ``S_in``: the sequences' entry states
    ``[N, H, d, d]`` or None; ``store``: a ``torch.distributed.Store`` shared by the ranks;
    ``group``: the process group (default group when None).  Every rank of the group must
    make the same calls in the same order (the call key is a per-process counter unless
    ``tag`` is given).  Returns ``parts.run``'s result; raises :class:`KcpError` on every
    surviving rank when a rank fails or does not arrive within ``timeout_s``."""
    import torch.distributed as dist

    parts = parts or gpu_parts()
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    tag = tag or f"kcp/{next(_calls)}"

    # 1. this rank's pair
    err = None
    try:
        M, St = parts.pairs(local)
        mine = f"ok:{tuple(M.shape)}:{M.dtype}"
    except Exception as e:  # reported to the other ranks, then re-raised here
        err, mine = e, "failed:" + type(e).__name__
    # 2. readiness, bounded: no collective is entered unless every rank is ready; a rank
    #    whose pair failed says so and leaves at once
    if err is not None:
        store.set(f"{tag}/{rank}", mine)
        raise KcpError(f"rank {rank}: its pair failed ({type(err).__name__}: {err})") from err
    posts = _post_and_wait(store, tag, rank, world, mine, timeout_s)
    failed = [r for r, p in enumerate(posts) if not p.startswith("ok:")]
    if failed:
        raise KcpError(f"rank(s) {failed} failed before the exchange")
    if len(set(posts)) != 1:
        raise KcpError(f"ranks disagree on the pairs' shapes: {posts}")
    # 3. one all-gather of the pairs (fixed size), into local tensors
    P = torch.stack([M, St]).contiguous()
    if world > 1:
        gathered = [torch.empty_like(P) for _ in range(world)]
        dist.all_gather(gathered, P, group=group)
    else:
        gathered = [P]
    # 4. local combine of the preceding ranks' pairs
    prev = torch.stack(gathered[:rank]) if rank > 0 else P.new_empty((0,) + tuple(P.shape))
    entry = parts.combine(prev[:, 0], prev[:, 1], S_in)
    # 5. this rank's rows from the true entry states
    return parts.run(local, entry)
