"""Kernel-only timing of the q8_1 prepass and every GEMM path over the named
workloads (7B-at-2K shapes and the token-count sweep), one JSON line each.

Each timing rotates through enough independent input sets that every launch
reads its inputs from HBM (the sets together exceed twice the 129 MB L2),
and uses CUDA events on the launching stream after warm-up.  The reported
kernel time replays the launches from a CUDA graph (no host launch cost);
the plain stream-launch time is reported beside it.

The path "q6k" times the q6_K x q8_1 GEMM (mmq_q6K_gemm) on q6_K weights
of the same shapes, repacked once to the device layout before timing.

Extra shapes: --shapes M:K:N,... (named shape_MxKxN); --pdl launches with
programmatic dependent launch (mmq_set_programmatic_launch).

  python -m q4_q8_int8_gb300.tools.sweep [--reps 50] [--paths auto,tc,mma_s8,small_m,q6k]
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math

import torch

import q4_q8_int8_gb300 as mmq
from q4_q8_int8_gb300 import build, synthetic

PATHS = {"auto": mmq.MMQ_PATH_AUTO, "tc": mmq.MMQ_PATH_TC, "mma_s8": mmq.MMQ_PATH_MMA_S8,
         "small_m": mmq.MMQ_PATH_SMALL_M, "tc_pair": mmq.MMQ_PATH_TC_PAIR, "tc_small": mmq.MMQ_PATH_TC_SMALL,
         "q6k": "q6k"}


def shapes(extra=()):
    for M, K, N in extra:
        yield f"shape_{M}x{K}x{N}", M, K, N
    for name in ("q_proj", "gate_up", "down"):
        M, K, N = synthetic.SHAPES[name]
        yield name, M, K, N
    for M in synthetic.SWEEP_M:
        yield f"sweep_M{M}", M, 4096, 4096


def time_gemm(M, K, N, path, reps, dev, graph=True):
    q6 = path == "q6k"
    set_bytes = N * K * (0.875 if q6 else 0.5625) + M * K * 1.25 + M * N * 4 + M * K * 4
    R = max(2, math.ceil(2 * 129e6 / set_bytes) + 1)
    R = min(R, 64)
    if q6:
        ws = [mmq.repack_q6K(synthetic.torch_q6K_weights(N, K, 100 + r, dev).view(-1), N, K) for r in range(R)]
    else:
        ws = [synthetic.torch_q4K_weights(N, K, 100 + r, dev).view(-1) for r in range(R)]
    xs = [synthetic.torch_activations(M, K, 200 + r, dev) for r in range(R)]
    aqs = [mmq.quantize_q8_1(x) for x in xs]
    Cs = [torch.empty((M, N), device=dev) for _ in range(R)]
    sp = mmq._stream_ptr()
    structs = [mmq.q8_1_struct(*aq) for aq in aqs]

    def gemm_call(r, stream_ptr):
        if q6:
            return mmq.mmq_q6K_gemm(structs[r], ctypes.c_void_p(ws[r].data_ptr()),
                                    ctypes.c_void_p(Cs[r].data_ptr()), M, N, K, stream_ptr)
        return mmq.mmq_q4K_gemm_path(structs[r], ctypes.c_void_p(ws[r].data_ptr()),
                                     ctypes.c_void_p(Cs[r].data_ptr()), M, N, K, path, stream_ptr)

    def launch(i):
        rc = gemm_call(i % R, sp)
        if rc:
            raise mmq.MMQError(rc, "gemm")

    def launch_q(i):
        r = i % R
        rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(xs[r].data_ptr()), M, K, structs[r], sp)
        if rc:
            raise mmq.MMQError(rc, "quantize")

    out = {}
    for label, fn in (("gemm", launch), ("prepass", launch_q)):
        for i in range(5):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(reps):
            fn(i)
        e1.record()
        torch.cuda.synchronize()
        out[label] = e0.elapsed_time(e1) / reps
        if not graph:
            out[label + "_graph"] = out[label]
            continue
        # device time without host launch cost: the same launches replayed from a CUDA graph
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            global_sp = mmq._stream_ptr(s)
            with torch.cuda.graph(g, stream=s):
                for i in range(reps):
                    r = i % R
                    if label == "gemm":
                        rc = gemm_call(r, global_sp)
                    else:
                        rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(xs[r].data_ptr()), M, K,
                                                   structs[r], global_sp)
                    if rc:
                        raise mmq.MMQError(rc, label)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        out[label + "_graph"] = e0.elapsed_time(e1) / reps
    if mmq.status() != 0:
        raise RuntimeError("device status error")
    return out, R


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=50)
    ap.add_argument("--paths", default="auto")
    ap.add_argument("--workloads", default="", help="comma-separated subset, e.g. q_proj,sweep_M1")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph timing (for profilers)")
    ap.add_argument("--shapes", default="", help="extra M:K:N shapes, comma-separated")
    ap.add_argument("--pdl", action="store_true")
    args = ap.parse_args()
    build.build()
    mmq.load_library()
    mmq.mmq_set_programmatic_launch(args.pdl)
    extra = [tuple(int(v) for v in sh.split(":")) for sh in args.shapes.split(",") if sh]
    dev = torch.device("cuda", 0)
    hbm = 6785.2
    only = set(w for w in args.workloads.split(",") if w)
    for name, M, K, N in shapes(extra):
        if (only or extra) and name not in only and not name.startswith("shape_"):
            continue
        for pname in args.paths.split(","):
            path = PATHS[pname]
            if path == mmq.MMQ_PATH_SMALL_M and M > mmq.SMALL_M_MAX:
                continue
            t, R = time_gemm(M, K, N, path, args.reps, dev, graph=not args.no_graph)
            ms = t["gemm_graph"]
            macs = M * N * K
            gbytes = (N * K * (0.875 if path == "q6k" else 0.5625) + M * K * 1.25 + M * N * 4) / 1e9
            print(json.dumps({
                "workload": name, "M": M, "K": K, "N": N, "path": pname,
                "gemm_us": ms * 1e3, "tmacs": macs / (ms * 1e-3) / 1e12,
                "us_per_gmac": ms * 1e3 / (macs / 1e9),
                "gemm_gbs": gbytes / (ms * 1e-3), "hbm_frac_of_measured": gbytes / (ms * 1e-3) / hbm,
                "gemm_us_stream_launch": t["gemm"] * 1e3,
                "prepass_us": t["prepass_graph"] * 1e3,
                "prepass_gbs": M * K * 5.25 / 1e9 / (t["prepass_graph"] * 1e-3),
                "rotating_sets": R}), flush=True)


if __name__ == "__main__":
    main()
