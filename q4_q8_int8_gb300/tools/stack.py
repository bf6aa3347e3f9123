"""The 7B-shaped prefill linear stack on one GPU: 32 layers x {q, k, v, o,
gate, up, down} at 2048 tokens, independent seeded q4_K weights per (layer,
GEMM) resident in HBM (3.64 GB), one q8_1 prepass per GEMM.  Prints one JSON
line with the stack time (prepasses included) as equivalent tokens/s and
TMAC/s, and the GEMM-only and prepass-only split.

Activations are drawn on the device per GEMM before timing; a pool of eight
activation sets per input width is reused round-robin during the timed
passes (every weight matrix is distinct, so nothing of the weight stream is
served from L2).

With --fused every GEMM writes its result as q8_1 from its epilogue
(mmq_q4K_gemm_q8_1 without the f32 output) and reads q8_1 activations that
were quantized once before timing: the stack as it runs when each GEMM's
output prepass is folded into the producing GEMM.

With --swiglu (implies --fused) each layer's gate and up weights are
interleaved once at set-up and run as one GEMM whose epilogue applies
silu(gate) * up and quantizes to q8_1 (mmq_q4K_gemm_swiglu_q8_1); that
output is the down projection's input, as in a SwiGLU FFN block.

  python -m q4_q8_int8_gb300.tools.stack [--passes 3] [--path auto] [--fused] [--swiglu]
"""
from __future__ import annotations

import argparse
import ctypes
import json

import torch

import q4_q8_int8_gb300 as mmq
from q4_q8_int8_gb300 import build, synthetic

PATHS = {"auto": mmq.MMQ_PATH_AUTO, "tc": mmq.MMQ_PATH_TC, "tc_pair": mmq.MMQ_PATH_TC_PAIR}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--passes", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--path", default="auto", choices=sorted(PATHS))
    ap.add_argument("--layers", type=int, default=synthetic.STACK_LAYERS)
    ap.add_argument("--fused", action="store_true")
    ap.add_argument("--swiglu", action="store_true")
    ap.add_argument("--pdl", action="store_true", help="programmatic dependent launch (mmq_set_programmatic_launch)")
    args = ap.parse_args()
    if args.swiglu:
        args.fused = True
    build.build()
    mmq.load_library()
    mmq.mmq_set_programmatic_launch(args.pdl)
    dev = torch.device("cuda", 0)
    M = synthetic.STACK_TOKENS
    path = PATHS[args.path]
    weights = []   # (K, N, bytes, kind); kind "glu": N = 2F interleaved gate / up rows
    names = [n for n, _, _ in synthetic.STACK_GEMMS]
    for layer in range(args.layers):
        pending = {}
        for g, (name, K, N) in enumerate(synthetic.STACK_GEMMS):
            ws, _ = synthetic.stack_seeds(layer, g)
            w = synthetic.torch_q4K_weights(N, K, ws, dev).view(-1)
            if args.swiglu and name in ("gate", "up"):
                pending[name] = w
                if len(pending) == 2:
                    weights.append((K, 2 * N, mmq.interleave_rows_q4K(pending["gate"], pending["up"], N, K), "glu"))
                    del pending
                    pending = {}
                continue
            weights.append((K, N, w, "down" if (args.swiglu and name == "down") else "gemm"))
    assert not args.swiglu or {"gate", "up", "down"} <= set(names)
    pool = {}
    for K in sorted({K for _, K, _ in synthetic.STACK_GEMMS}):
        xs = []
        for i in range(8):
            _, xseed = synthetic.stack_seeds(i, 0 if K == 4096 else 6)
            xs.append(synthetic.torch_activations(M, K, xseed, dev, 0.01))
        pool[K] = (xs, [mmq.empty_q8_1(M, K, dev) for _ in xs])
    Ns = sorted({N for _, _, N in synthetic.STACK_GEMMS})
    outs = {N: torch.empty((M, N), device=dev) for N in Ns}
    outs_q8 = {N: mmq.q8_1_struct(*mmq.empty_q8_1(M, N, dev)) for N in Ns}
    F = max(Ns)
    glu_out = mmq.q8_1_struct(*mmq.empty_q8_1(M, F, dev))   # the down projection's input
    sp = mmq._stream_ptr()
    structs = {K: [mmq.q8_1_struct(*aq) for aq in pool[K][1]] for K in pool}
    if args.fused:   # activations quantized once, outside the timed passes
        for K in pool:
            for x, aqs in zip(pool[K][0], structs[K]):
                rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(x.data_ptr()), M, K, aqs, sp)
                if rc:
                    raise mmq.MMQError(rc, "quantize")

    def one_pass(ev=None):
        for i, (K, N, w, kind) in enumerate(weights):
            x = pool[K][0][i % 8]
            aqs = glu_out if kind == "down" else structs[K][i % 8]
            if ev is not None:
                ev[i][0].record()
            if not args.fused:
                rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(x.data_ptr()), M, K, aqs, sp)
                if rc:
                    raise mmq.MMQError(rc, "quantize")
            if ev is not None:
                ev[i][1].record()
            if kind == "glu":
                rc = mmq.mmq_q4K_gemm_swiglu_q8_1(aqs, ctypes.c_void_p(w.data_ptr()), None, glu_out, M, N // 2,
                                                  K, sp)
            elif args.fused:
                rc = mmq.mmq_q4K_gemm_q8_1(aqs, ctypes.c_void_p(w.data_ptr()), None, outs_q8[N], M, N, K, sp)
            else:
                rc = mmq.mmq_q4K_gemm_path(aqs, ctypes.c_void_p(w.data_ptr()),
                                           ctypes.c_void_p(outs[N].data_ptr()), M, N, K, path, sp)
            if rc:
                raise mmq.MMQError(rc, "gemm")
            if ev is not None:
                ev[i][2].record()

    for _ in range(args.warmup):
        one_pass()
    torch.cuda.synchronize()
    t_stack, t_gemm, t_pre = [], [], []
    for _ in range(args.passes):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        one_pass()
        e1.record()
        torch.cuda.synchronize()
        t_stack.append(e0.elapsed_time(e1))
    # a separate pass with per-launch events for the GEMM / prepass split
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in weights]
    one_pass(ev)
    torch.cuda.synchronize()
    t_pre = sum(a.elapsed_time(b) for a, b, _ in ev)
    t_gemm = sum(b.elapsed_time(c) for _, b, c in ev)
    if mmq.status() != 0:
        raise RuntimeError("device status error")
    macs = sum(M * K * N for K, N, _, _ in weights)
    best = min(t_stack)
    print(json.dumps({
        "workload": f"7B prefill stack: {args.layers} layers x (q,k,v,o 4096x4096; gate,up 4096->11008; "
                    f"down 11008->4096), M={M}",
        "path": args.path, "passes": args.passes, "fused_requantize": args.fused, "fused_swiglu": args.swiglu,
        "programmatic_launch": args.pdl,
        "stack_ms": {"min": best, "median": sorted(t_stack)[len(t_stack) // 2], "max": max(t_stack)},
        "equivalent_tok_s": M / (best * 1e-3),
        "tmacs_with_prepass": macs / (best * 1e-3) / 1e12,
        "gemm_only_ms": t_gemm, "gemm_only_tmacs": macs / (t_gemm * 1e-3) / 1e12,
        "prepass_ms": t_pre, "gmac": macs / 1e9,
        "weights_gb": sum(w.numel() for _, _, w, _ in weights) / 1e9,
    }))


if __name__ == "__main__":
    main()
