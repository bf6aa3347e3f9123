"""One decode step of the 7B-shaped linear stack on one GPU: 32 layers x {q,
k, v, o 4096->4096; gate, up 4096->11008; down 11008->4096} at a few tokens
(default 1), each GEMM preceded by its q8_1 prepass, all 224 weight matrices
(3.64 GB of q4_K) distinct and resident in HBM.  A GEMM's output is the next
prepass's input wherever the widths allow (so consecutive kernels really
depend on each other); elsewhere the input comes from a pool.

The step is captured once in a CUDA graph and replayed; with --pdl the
prepass and GEMM kernels are launched with programmatic dependent launch
(mmq_set_programmatic_launch), so each starts streaming its weights while
the previous kernel finishes.  With --fused every GEMM writes its result as
q8_1 (mmq_q4K_gemm_q8_1) and the next GEMM reads it with no prepass between
them: one kernel per GEMM for 1 to 4 tokens (q8_1 out of the dot-product
kernel's epilogue), a GEMM and a quantize pass for more.  Prints one JSON line: step time, tokens/s,
and the weight stream's rate against the measured HBM copy bandwidth.

  python -m q4_q8_int8_gb300.tools.decode [--tokens 1] [--pdl] [--fused] [--replays 20]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os

import torch

import q4_q8_int8_gb300 as mmq
from q4_q8_int8_gb300 import build, synthetic


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--layers", type=int, default=synthetic.STACK_LAYERS)
    ap.add_argument("--replays", type=int, default=20)
    ap.add_argument("--pdl", action="store_true")
    ap.add_argument("--fused", action="store_true")
    args = ap.parse_args()
    build.build()
    mmq.load_library()
    dev = torch.device("cuda", 0)
    M = args.tokens
    mmq.mmq_set_programmatic_launch(args.pdl)
    gemms = []
    for layer in range(args.layers):
        for g, (_, K, N) in enumerate(synthetic.STACK_GEMMS):
            ws, xs = synthetic.stack_seeds(layer, g)
            gemms.append((K, N, synthetic.torch_q4K_weights(N, K, ws, dev).view(-1)))
    widths = sorted({K for K, _, _ in gemms} | {N for _, N, _ in gemms})
    pool = {k: synthetic.torch_activations(M, k, 9000 + k, dev) for k in widths}
    outs = [torch.empty((M, N), device=dev) for _, N, _ in gemms]
    q8 = {k: mmq.q8_1_struct(*mmq.empty_q8_1(M, k, dev)) for k in widths}
    # --fused: q8_1 pools (the pool's activations quantized once, outside the
    # step) and two ping-pong q8_1 outputs per width
    qpool_t = {k: mmq.quantize_q8_1(pool[k]) for k in widths}   # keeps the tensors alive
    torch.cuda.synchronize()
    qpool = {k: mmq.q8_1_struct(*v) for k, v in qpool_t.items()}
    qbufs = [{k: mmq.empty_q8_1(M, k, dev) for k in widths} for _ in range(2)]
    qout = [{k: mmq.q8_1_struct(*b[k]) for k in widths} for b in qbufs]
    stream = torch.cuda.Stream(dev)

    def step():
        sp = mmq._stream_ptr(stream)
        prev = None
        qprev, N_prev = None, 0
        for i, (K, N, w) in enumerate(gemms):
            x = prev if (prev is not None and prev.shape[1] == K) else pool[K]
            if args.fused:
                # q8_1 in: the previous GEMM's q8_1 output where the widths chain, else
                # a prequantized pool entry; q8_1 out (and no f32 result for M <= 4)
                src = qprev if (qprev is not None and N_prev == K) else qpool[K]
                rc = mmq.mmq_q4K_gemm_q8_1(src, ctypes.c_void_p(w.data_ptr()),
                                           ctypes.c_void_p(0 if M <= 4 else outs[i].data_ptr()),
                                           qout[i % 2][N], M, N, K, sp)
                qprev, N_prev = qout[i % 2][N], N
            else:
                rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(x.data_ptr()), M, K, q8[K], sp)
                rc |= mmq.mmq_q4K_gemm(q8[K], ctypes.c_void_p(w.data_ptr()),
                                       ctypes.c_void_p(outs[i].data_ptr()), M, N, K, sp)
            if rc:
                raise mmq.MMQError(rc, "decode step")
            prev = outs[i]

    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.replays):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    if mmq.status(stream) != 0:
        raise RuntimeError("device status error")
    us = e0.elapsed_time(e1) * 1e3 / args.replays
    wbytes = sum(w.numel() for _, _, w in gemms)
    hbm = 6785.0
    p = os.path.join(os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))),
                     "MEASURED_PEAKS.json")
    if os.path.exists(p):
        hbm = json.load(open(p))["hbm_gbs"]
    nk = (1 if args.fused and M <= 4 else 2) * len(gemms)
    print(json.dumps({
        "workload": f"7B decode step: {args.layers} layers x 7 GEMMs, {M} token(s), "
                    + ("q8_1 out of each GEMM" if args.fused else "prepass per GEMM"),
        "programmatic_launch": args.pdl, "fused_prepass": args.fused, "kernels": nk,
        "step_us": us, "tokens_per_s": M / (us * 1e-6),
        "weights_gb": wbytes / 1e9, "weight_stream_gbs": wbytes / (us * 1e-6) / 1e9,
        "frac_of_measured_hbm": wbytes / (us * 1e-6) / 1e9 / hbm,
        "us_per_kernel": us / nk,
    }))


if __name__ == "__main__":
    main()
