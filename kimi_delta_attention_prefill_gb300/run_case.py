"""Run one workload through the library a few times (for profilers and quick checks).

    python -m kimi_delta_attention_prefill_gb300.run_case --workload prefill_8k --heads 16 --iters 3
    python -m kimi_delta_attention_prefill_gb300.run_case --workload prefill_8k --gated   # + output stage

Prints the mean CUDA-event time per call; exits non-zero if the library reports an error.
"""
from __future__ import annotations

import argparse

import torch

import kimi_delta_attention_prefill_gb300 as kda
from kimi_delta_attention_prefill_gb300 import inputs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="prefill_8k", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--heads", type=int, default=None, help="override the head count")
    ap.add_argument("--tokens", type=int, default=None, help="override the length of a single-sequence prefill")
    ap.add_argument("--segments", type=int, default=0, help="prefill segment count (0 = library's choice)")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--gated", action="store_true", help="prefill with the fused output stage")
    args = ap.parse_args()
    over = {}
    if args.heads:
        over["H"] = args.heads
    if args.tokens:
        over["lengths"] = [args.tokens]
    x = inputs.make_workload(args.workload, device="cuda", **over)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if inputs.WORKLOADS[args.workload]["kind"] == "decode":
        S = x.S0.clone()
        nc = None if x.n_commit is None else x.n_commit.cuda()
        run = lambda: kda.decode(x.q, x.k, x.v, x.g, x.beta, S, n_commit=nc, dev_status=status)
    else:
        cu = x.cu_seqlens.cuda()
        off = None if x.ckpt_off is None else x.ckpt_off.cuda()
        pos = None if x.ckpt_pos is None else x.ckpt_pos.cuda()
        S0 = x.S0
        kw = {}
        if args.gated:
            gate, w = inputs.make_output_stage(x.q.shape[0], x.q.shape[1], device="cuda")
            kw = dict(gate=gate, norm_weight=w)
        run = lambda: kda.prefill(x.q, x.k, x.v, x.g, x.beta, cu, S_in=S0, ckpt_off=off, ckpt_pos=pos,
                                  n_segments=args.segments, dev_status=status, **kw)
    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    st = int(status.item())
    print(f"{args.workload}: {e0.elapsed_time(e1) / args.iters * 1e3:.1f} us per call, status {st}")
    if st != 0:
        raise SystemExit(f"device status {kda.status_string(st)}")


if __name__ == "__main__":
    main()
