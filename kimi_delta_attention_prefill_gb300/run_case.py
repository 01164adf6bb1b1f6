"""Run one workload through the library a few times (for profilers and quick checks).

    python -m kimi_delta_attention_prefill_gb300.run_case --workload prefill_8k --heads 16 --iters 3
    python -m kimi_delta_attention_prefill_gb300.run_case --workload prefill_8k --gated   # + output stage
    python -m kimi_delta_attention_prefill_gb300.run_case --workload verify --fused        # decode front end
    python -m kimi_delta_attention_prefill_gb300.run_case --workload decode --paged        # states in pages

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
    ap.add_argument("--n-seq", type=int, default=1, help="with --tokens: this many sequences of that length")
    ap.add_argument("--segments", type=int, default=0, help="prefill segment count (0 = library's choice)")
    ap.add_argument("--n-tok", type=int, default=None, help="override the tokens of a decode / verify step")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--gated", action="store_true", help="prefill with the fused output stage")
    ap.add_argument("--fused", action="store_true",
                    help="decode from projected inputs (kda_decode_fused: width-4 conv + SiLU, output stage)")
    ap.add_argument("--paged", action="store_true",
                    help="decode with the states scattered in a page pool (kda_decode_paged, copy to fresh pages)")
    args = ap.parse_args()
    over = {}
    if args.heads:
        over["H"] = args.heads
    if args.tokens:
        over["lengths"] = [args.tokens] * args.n_seq
    if args.n_tok:
        over["n_tok"] = args.n_tok
    x = inputs.make_workload(args.workload, device="cuda", **over)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if inputs.WORKLOADS[args.workload]["kind"] == "decode":
        S = x.S0.clone()
        nc = None if x.n_commit is None else x.n_commit.cuda()
        B, n_tok, H = x.q.shape[0], x.q.shape[1], x.q.shape[2]
        if args.fused:
            w = inputs.WORKLOADS[args.workload]
            fx = inputs.make_decode_frontend(B, n_tok, H, W=4, seed=w["seed"], device="cuda",
                                             commit=w.get("commit", "all"))
            fS, fc = fx.S0.clone(), fx.conv_cache.clone()
            fnc = None if fx.n_commit is None else fx.n_commit.cuda()
            run = lambda: kda.decode_fused(fx.qp, fx.kp, fx.vp, fx.conv_w, fc, fx.z, fx.a_log, fx.b, fS, n_commit=fnc,
                                           conv_act="silu", gate=fx.gate, norm_weight=fx.norm_weight,
                                           dev_status=status)
        elif args.paged:
            n_units = B * H
            pin, pout = inputs.make_page_tables([n_units, n_units], 2 * n_units + 1024, seed=5)
            pool = torch.zeros((2 * n_units + 1024, 128, 128), dtype=torch.float32, device="cuda")
            pool[pin.long().cuda()] = x.S0.reshape(-1, 128, 128)
            pin, pout = pin.cuda(), pout.cuda()
            run = lambda: kda.decode_paged(x.q, x.k, x.v, x.g, x.beta, pool, pin, pout, n_commit=nc, dev_status=status)
        else:
            run = lambda: kda.decode(x.q, x.k, x.v, x.g, x.beta, S, n_commit=nc, dev_status=status)
    else:
        cu = x.cu_seqlens.cuda()
        off = None if x.ckpt_off is None else x.ckpt_off.cuda()
        pos = None if x.ckpt_pos is None else x.ckpt_pos.cuda()
        S0 = x.S0
        kw = {}
        if args.gated:
            gate, w = inputs.make_output_stage(x.q.shape[0], x.q.shape[1], seed=1, device="cuda")
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
