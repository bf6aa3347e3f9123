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
them: one kernel per GEMM up to 64 tokens (q8_1 out of the few-token
kernels' epilogues).  Prints one JSON line: step time, tokens/s,
and the weight stream's rate against the measured HBM copy bandwidth.

With --model the step has a transformer layer's structure instead: q, k
and v as one 4096 -> 12288 GEMM (their rows concatenated), o, gate and up as
one 4096 -> 2 x 11008 GEMM on interleaved rows with the SwiGLU and the q8_1
quantization in its epilogue (mmq_q4K_gemm_swiglu_q8_1), and down; a q8_1
prepass before q/k/v, o and gate/up.  Attention, the norms and the residual
adds are not part of this library: o reads a resident activation in place
of the attention output, and each prepass reads the previous GEMM's f32
output in place of the normalized residual.  Same 3.64 GB of weights,
7 kernels per layer.

  python -m q4_q8_int8_gb300.tools.decode [--tokens 1] [--pdl] [--fused | --model] [--replays 20]
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
    ap.add_argument("--model", action="store_true")
    args = ap.parse_args()
    build.build()
    mmq.load_library()
    dev = torch.device("cuda", 0)
    M = args.tokens
    mmq.mmq_set_programmatic_launch(args.pdl)
    gemms = []
    # --model: per layer q|k|v (4096 -> 12288), o, gate|up interleaved (4096 -> 2 x 11008), down
    shapes = ((4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)) if args.model else \
        tuple((K, N) for _, K, N in synthetic.STACK_GEMMS)
    for layer in range(args.layers):
        for g, (K, N) in enumerate(shapes):
            ws, xs = synthetic.stack_seeds(layer, g)
            gemms.append((K, N, synthetic.torch_q4K_weights(N, K, ws, dev).view(-1)))
    widths = sorted({K for K, _, _ in gemms} | {N for _, N, _ in gemms} | {11008})
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
    P = lambda t: ctypes.c_void_p(t.data_ptr())

    def model_step():
        sp = mmq._stream_ptr(stream)
        x = pool[4096]
        rc = 0
        for layer in range(args.layers):
            (_, _, w_qkv), (_, _, w_o), (_, _, w_gu), (_, _, w_down) = gemms[4 * layer:4 * layer + 4]
            o_qkv, o_o, _, o_down = outs[4 * layer:4 * layer + 4]
            rc |= mmq.mmq_quantize_q8_1(P(x), M, 4096, q8[4096], sp)
            rc |= mmq.mmq_q4K_gemm(q8[4096], P(w_qkv), P(o_qkv), M, 12288, 4096, sp)
            rc |= mmq.mmq_quantize_q8_1(P(pool[4096]), M, 4096, q8[4096], sp)   # attention output stand-in
            rc |= mmq.mmq_q4K_gemm(q8[4096], P(w_o), P(o_o), M, 4096, 4096, sp)
            rc |= mmq.mmq_quantize_q8_1(P(o_o), M, 4096, q8[4096], sp)
            rc |= mmq.mmq_q4K_gemm_swiglu_q8_1(q8[4096], P(w_gu), None, q8[11008], M, 11008, 4096, sp)
            rc |= mmq.mmq_q4K_gemm(q8[11008], P(w_down), P(o_down), M, 4096, 11008, sp)
            x = o_down
        if rc:
            raise mmq.MMQError(rc, "decode step")

    def step():
        if args.model:
            return model_step()
        sp = mmq._stream_ptr(stream)
        prev = None
        qprev, N_prev = None, 0
        for i, (K, N, w) in enumerate(gemms):
            x = prev if (prev is not None and prev.shape[1] == K) else pool[K]
            if args.fused:
                # q8_1 in: the previous GEMM's q8_1 output where the widths chain, else
                # a prequantized pool entry; q8_1 out (and no f32 result up to 64 tokens)
                src = qprev if (qprev is not None and N_prev == K) else qpool[K]
                rc = mmq.mmq_q4K_gemm_q8_1(src, ctypes.c_void_p(w.data_ptr()),
                                           ctypes.c_void_p(0 if M <= 64 else outs[i].data_ptr()),
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
    nk = 7 * args.layers if args.model else (1 if args.fused and M <= 64 else 2) * len(gemms)
    print(json.dumps({
        "workload": (f"7B decode step, layer structure: {args.layers} x (qkv, o, gate|up + SwiGLU, down), "
                     f"{M} token(s)") if args.model else
                    (f"7B decode step: {args.layers} layers x 7 GEMMs, {M} token(s), "
                     + ("q8_1 out of each GEMM" if args.fused else "prepass per GEMM")),
        "programmatic_launch": args.pdl, "fused_prepass": args.fused, "kernels": nk,
        "step_us": us, "tokens_per_s": M / (us * 1e-6),
        "weights_gb": wbytes / 1e9, "weight_stream_gbs": wbytes / (us * 1e-6) / 1e9,
        "frac_of_measured_hbm": wbytes / (us * 1e-6) / 1e9 / hbm,
        "us_per_kernel": us / nk,
    }))


if __name__ == "__main__":
    main()
