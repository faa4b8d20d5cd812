"""Profiling harness: runs one entry point of the library on a named synthetic case a
few times, so that a profiler can capture a handful of launches of one kernel.

  python -m gated_delta_rule_53_gb300.profile {prefill_8k,prefill_8k_gate,prefill_2k,varlen_small,long_16k,
                                               decode_64,decode_16,frontend_8k,gates_8k,bwd_8k,bwd_2k} [--iters N]

Cases (all inputs larger than the 129 MB L2, a few GB on the device at most):
  prefill_8k   kda_chunk_fwd, 1 x 8192 tokens x 96 heads, bf16
  prefill_8k_gate  the same with a bf16 N(0, 1) sigmoid output gate (the long workload's epilogue)
  prefill_2k   kda_chunk_fwd, 1 x 2048 tokens x 96 heads, bf16
  varlen_small kda_chunk_fwd, 4 packed sequences (1500, 3000, 2100, 2600 tokens) x 96 heads, bf16, initial
               states N(0, 0.02): the packed path of the 32-sequence workload at about 1/57 of its tokens
  long_16k     kda_chunk_fwd_frontend with the sigmoid output gate, 16384 tokens x 96 heads from raw bf16 rows:
               the long workload's path at 1/16 of its tokens (one range of 256 chunk rows, overlapped)
  decode_64    kda_recurrent_step, 64 sequences x 96 heads
  decode_16    kda_recurrent_step, 16 sequences x 96 heads
  frontend_8k  kda_shortconv_l2norm, 8192 tokens x 96 heads, bf16 out
  gates_8k     kda_gate_generator, x 8192 x 7168 -> 96 x 128 gate channels, rank 128 (bench.py's sizes)
  bwd_8k       kda_chunk_bwd of prefill_8k (bf16 inputs and dL/do), as bench.py's backward leg
  bwd_2k       kda_chunk_bwd, 1 x 2048 tokens x 96 heads
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import torch

    import gated_delta_rule_53_gb300 as kda
    import kda_synth as ks
    from kda_synth.device import fill_device

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["prefill_8k", "prefill_8k_gate", "prefill_2k", "varlen_small", "long_16k",
                                     "decode_64", "decode_16", "frontend_8k", "gates_8k", "bwd_8k", "bwd_2k"])
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if args.case.startswith("prefill") or args.case.startswith("bwd"):
        T = 8192 if "8k" in args.case else 2048
        w = ks.Workload(args.case, "prefill", 53002, H=96, lengths=[T])
        q = fill_device(w.seed, ks.TID_Q, ks.UNIT_GROUPS, (T, 96, 128), "bf16", 0.0, 128.0, device=dev)
        k = fill_device(w.seed, ks.TID_K, ks.UNIT_GROUPS, (T, 96, 128), "bf16", 0.0, 128.0, device=dev)
        v = fill_device(w.seed, ks.TID_V, ks.NORMAL, (T, 96, 128), "bf16", device=dev)
        g = fill_device(w.seed, ks.TID_G, w.g_kind, (T, 96, 128), "f32", device=dev)
        b = fill_device(w.seed, ks.TID_BETA, ks.SIGMOID, (T, 96), "f32", device=dev)
        fn = lambda: kda.kda_chunk_fwd(q, k, v, g, b)
        if args.case == "prefill_8k_gate":
            gate = fill_device(w.seed, ks.TID_GATE, ks.NORMAL, (T, 96 * 128), "bf16", device=dev)
            fn = lambda: kda.kda_chunk_fwd(q, k, v, g, b, out_gate=gate)
        if args.case.startswith("bwd"):
            do = fill_device(w.seed, ks.TID_DO, ks.NORMAL, (T, 96, 128), "bf16", device=dev)
            ws = torch.empty(kda.kda_chunk_bwd_workspace_size(1, T, 96), dtype=torch.uint8, device=dev)
            fn = lambda: kda.kda_chunk_bwd(q, k, v, g, b, do, workspace=ws)
    elif args.case == "varlen_small":
        w = ks.Workload(args.case, "prefill", 53004, H=96, lengths=[1500, 3000, 2100, 2600], init_state_std=0.02)
        T, N = w.T, w.N
        q = fill_device(w.seed, ks.TID_Q, ks.UNIT_GROUPS, (T, 96, 128), "bf16", 0.0, 128.0, device=dev)
        k = fill_device(w.seed, ks.TID_K, ks.UNIT_GROUPS, (T, 96, 128), "bf16", 0.0, 128.0, device=dev)
        v = fill_device(w.seed, ks.TID_V, ks.NORMAL, (T, 96, 128), "bf16", device=dev)
        g = fill_device(w.seed, ks.TID_G, w.g_kind, (T, 96, 128), "f32", device=dev)
        b = fill_device(w.seed, ks.TID_BETA, ks.SIGMOID, (T, 96), "f32", device=dev)
        s0 = fill_device(w.seed, ks.TID_STATE, ks.NORMAL, (N, 96, 128, 128), "f32", 0.0, 0.02, device=dev)
        cu = torch.from_numpy(w.cu_seqlens()).to(dev)
        fn = lambda: kda.kda_chunk_fwd(q, k, v, g, b, s0, cu)
    elif args.case == "long_16k":
        T, C = 16384, 96 * 128
        w = ks.Workload(args.case, "frontend", 53005, H=96, lengths=[T], g_kind=ks.NEG_SOFTPLUS5)
        xs = [fill_device(w.seed, t, ks.NORMAL, (T, C), "bf16", device=dev) for t in (1, 2, 3)]
        cw = fill_device(w.seed, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25, device=dev)
        g = fill_device(w.seed, ks.TID_G, w.g_kind, (T, 96, 128), "f32", device=dev)
        b = fill_device(w.seed, ks.TID_BETA, ks.SIGMOID, (T, 96), "f32", device=dev)
        gate = fill_device(w.seed, ks.TID_GATE, ks.NORMAL, (T, C), "bf16", device=dev)
        fn = lambda: kda.kda_chunk_fwd_frontend(*xs, cw, g, b, 96, out_gate=gate)
    elif args.case.startswith("decode"):
        N = 64 if args.case == "decode_64" else 16
        w = ks.Workload(args.case, "decode", 53003, H=96, lengths=[1] * N, init_state_std=0.02)
        C = 96 * 128
        xs = [fill_device(w.seed, t, ks.NORMAL, (N, C), "bf16", device=dev) for t in (1, 2, 3)]
        cw = fill_device(w.seed, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25, device=dev)
        g = fill_device(w.seed, ks.TID_G, w.g_kind, (N, 96, 128), "f32", device=dev)
        b = fill_device(w.seed, ks.TID_BETA, ks.SIGMOID, (N, 96), "f32", device=dev)
        st = fill_device(w.seed, ks.TID_STATE, ks.NORMAL, (N, 96, 128, 128), "f32", 0.0, 0.02, device=dev)
        cs = fill_device(w.seed, ks.TID_CONV_STATE, ks.NORMAL, (N, 3, 3 * C), "bf16", device=dev)
        fn = lambda: kda.kda_recurrent_step(*xs, cw, g, b, st, cs)
    elif args.case == "gates_8k":
        T, hid, H, d, rk = 8192, 7168, 96, 128, 128
        gen = torch.Generator(device=dev).manual_seed(53007)
        x = torch.randn(T, hid, device=dev, generator=gen).to(torch.bfloat16)
        wga = (torch.randn(H * d + rk, hid, device=dev, generator=gen) / hid ** 0.5).to(torch.bfloat16)
        wgb = (torch.randn(H * d, rk, device=dev, generator=gen) / rk ** 0.5).to(torch.bfloat16)
        ah = torch.randn(H, device=dev, generator=gen)
        fn = lambda: kda.kda_gate_generator(x, wga, wgb, ah, H, d)
    else:
        T, C = 8192, 96 * 128
        xs = [fill_device(53005, t, ks.NORMAL, (T, C), "bf16", device=dev) for t in (1, 2, 3)]
        cw = fill_device(53005, ks.TID_CONV_W, ks.NORMAL, (3 * C, 4), "bf16", 0.0, 0.25, device=dev)
        fn = lambda: kda.kda_shortconv_l2norm(*xs, cw, 96)
    for _ in range(args.iters):
        fn()
    torch.cuda.synchronize()
    print(f"{args.case}: {args.iters} iterations ok")


if __name__ == "__main__":
    main()
