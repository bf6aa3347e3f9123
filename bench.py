#!/usr/bin/env python3
"""Benchmark of the q4_K x q8_1 MMQ hot path on GB300.

One step = the whole hot path over one batch: the q8_1 quantize prepass of
the activations followed by the q4_K x q8_1 GEMM, on the 7B attention
q-projection at 2K-token prefill (M=2048 tokens, K=4096, N=4096), seeded
synthetic inputs.  Metric: TMAC/s = M*N*K / step time / 1e12 (higher is
better), with us/GMAC and the GEMM-only figures alongside.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

Under torchrun each rank runs its own independent problem on its own GPU
(weak scaling, no data-path collective); rank 0 prints one JSON line with
the max time over ranks.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload.

After the contract line's timed region, and outside it, rank 0 adds:
  "sweep"  kernel-only GEMM times of the other configurations (the FFN
           GEMMs at 2K tokens, the token-count sweep at 4096 x 4096 and the
           few-token decode shapes), each replayed from a CUDA graph over
           rotating inputs larger than twice the L2, with t_roof / t;
           "sweep_q6k" the same for q6_K weights;
  "stack"  the 32-layer 7B prefill linear stack (224 GEMMs, a prepass each)
           as equivalent tokens per second;
  "clocks" sampled from the warm-up to the end of a ~1 s soak of the same
           step loop, so that it holds many samples under load.
`--measure-peaks` compiles bench_peaks.cu (under _build/) and prints the
instruction-rate peaks recorded in profiles/peaks.json.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {"q_proj": (2048, 4096, 4096)}
PATH_NAMES = ("auto", "mma_s8", "tc", "small_m", "sb")
# "sb": the step runs the tensor-core prepass (q8_1 plus the operand plane) and
# the super-block GEMM on it (mmq_quantize_q8_1_tcop + mmq_q4K_gemm_tcop).
SB = "sb"
# A timed region shorter than this is held to the burst tensor peak, a longer
# one to the sustained peak (the GPU settles at its power cap within seconds).
SUSTAINED_AFTER_S = 1.0
L2_BYTES = 129e6
METRIC = "q4_K x q8_1 GEMM TMAC/s at 7B@2K (q-proj 2048x4096x4096), prepass included"
UNIT = "TMAC/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default="q_proj", choices=sorted(WORKLOADS))
    ap.add_argument("--path", default="auto", choices=sorted(PATH_NAMES))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-control", action="store_true", help="skip the dequantize-then-dense control timing")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch (mmq_set_programmatic_launch(0))")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="target seconds for the whole --impl reference run")
    ap.add_argument("--no-sweep", action="store_true", help="skip the extra configurations' kernel sweep")
    ap.add_argument("--no-stack", action="store_true", help="skip the 32-layer stack")
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="seconds of the step loop run after the timed region for the clock record")
    ap.add_argument("--shape", default=None, metavar="M:K:N",
                    help="profiling mode: run one GEMM shape --launches times on --path (or the q6_K kernels "
                         "with --weights q6k) and exit; no timing line (a target for ncu captures)")
    ap.add_argument("--weights", default="q4k", choices=["q4k", "q6k"])
    ap.add_argument("--launches", type=int, default=5)
    ap.add_argument("--measure-peaks", action="store_true",
                    help="compile and run bench_peaks.cu (instruction-rate peaks) and exit")
    ap.add_argument("--oracle-table", action="store_true",
                    help="with --impl reference: time the oracle's prepass and GEMM per configuration "
                         "(bounded row samples, extrapolated per row) instead of the contract line")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(vals, world, device=None):
    """Each value's maximum over all ranks (the slowest rank sets the job
    time); the values themselves when world == 1."""
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def whole_job_tmacs(macs_per_rank, world, max_ms):
    """Whole-job throughput: every rank's independent problem, over the
    slowest rank's time."""
    return macs_per_rank * world / (max_ms * 1e-3) / 1e12


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples the SM clock and clock-event reasons while active: through
    NVML (read-only queries, every 2 ms) when libnvidia-ml is present, else
    nvidia-smi every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, gpu_index: int, pci_bus_id: str | None = None):
        self.gpu_index = gpu_index
        self.pci_bus_id = pci_bus_id
        self.proc = None
        self.lines = []
        self.t = None
        self.nvml = None
        self.samples = []
        self.running = False

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.pci_bus_id:
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci_bus_id.encode(), ctypes.byref(h)) == 0
        if not ok:
            n = ctypes.c_uint()
            if lib.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0 or n.value != 1:
                return None
            if lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                return None
        return lib, h

    def _nvml_loop(self):
        import ctypes
        lib, h = self.nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while self.running:
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0):
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(0.002)

    def start(self):
        try:
            self.nvml = self._nvml_open()
        except OSError:
            self.nvml = None
        if self.nvml:
            self.running = True
            self.t = threading.Thread(target=self._nvml_loop, daemon=True)
            self.t.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.nvml:
            self.running = False
            self.t.join(timeout=2)
            sm = [c for c, _, _ in self.samples]
            reasons = set()
            for _, _, r in self.samples:
                for name, bit in self.BITS.items():
                    if r & bit:
                        reasons.add(name)
            return {"sm_mhz": float(np.median(sm)) if sm else None,
                    "sm_max_mhz": max(m for _, m, _ in self.samples) if self.samples else None,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml, 2 ms"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 200 ms"}


# ------------------------------------------------------------------ roofline
def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "q4_q8_int8_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def microbench_peaks():
    with open(os.path.join(ROOT, "profiles", "peaks.json")) as f:
        return json.load(f)


def recorded_traffic(kernel_key, src_hash):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("src_hash") != src_hash:
        return None
    return e.get("bytes_per_launch")


# ----------------------------------------------------------------- CPU leg
def cpu_oracle_sample(M, K, N, target_s, x, blk):
    """Time the oracle (quantize + blockwise GEMM) on the first m rows of the
    workload, m sized for about target_s seconds; returns (TMAC/s, m, secs, cores)."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    m = 1
    while True:
        t0 = time.perf_counter()
        q, da, sa = oracle.quantize_q8_1(x[:m])
        oracle.gemm(q, da, sa, blk, N, want_bound=False)
        dt = time.perf_counter() - t0
        if dt >= target_s or m >= M:
            break
        grow = max(2, int(target_s / max(dt, 1e-3) * 0.9))
        m = min(M, m * grow)
    return m * N * K / dt / 1e12, m, dt, cores


def _oracle_rows_timed(fn, M, target_s):
    """Time fn(m) on growing row counts m until it takes target_s or m == M;
    returns (seconds for m rows, m)."""
    m = 1
    while True:
        t0 = time.perf_counter()
        fn(m)
        dt = time.perf_counter() - t0
        if dt >= target_s or m >= M:
            return dt, m
        m = min(M, m * max(2, int(target_s / max(dt, 1e-3) * 0.9)))


def run_oracle_table(args):
    """The oracle's prepass and GEMM per configuration on this host's cores,
    on row samples of about args.cpu_seconds each; a sample smaller than the
    configuration is scaled per row and labelled extrapolated.  The 7B stack
    (32 layers x q, k, v, o, gate, up, down, a prepass per GEMM) is the sum
    of its GEMMs' timings x 32, labelled extrapolated."""
    from q4_q8_int8_gb300 import synthetic
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    items = [("tiny", None), ("q_proj", None), ("gate_up", None), ("down", None)]
    items += [("sweep", m) for m in synthetic.SWEEP_M]
    per = {}
    for name, msweep in items:
        x, blk, N = synthetic.config_inputs(name, msweep)
        M, K = x.shape
        tq, mq = _oracle_rows_timed(lambda m: oracle.quantize_q8_1(x[:m]), M, args.cpu_seconds / 4)
        q, da, sa = oracle.quantize_q8_1(x)
        tg, mg = _oracle_rows_timed(lambda m: oracle.gemm(q[:m], da[:m], sa[:m], blk, N, want_bound=False),
                                    M, args.cpu_seconds)
        prep_s, gemm_s = tq * M / mq, tg * M / mg
        label = name if msweep is None else f"sweep_M{msweep}"
        per[label] = (prep_s, gemm_s)
        print(json.dumps({"impl": "reference-table", "config": label, "M": M, "K": K, "N": N,
                          "prepass_s": prep_s, "gemm_s": gemm_s,
                          "gemm_tmacs": M * N * K / gemm_s / 1e12, "rows_timed": {"prepass": mq, "gemm": mg},
                          "extrapolated": bool(mq < M or mg < M), "cores": cores}), flush=True)
    layer = 4 * sum(per["q_proj"]) + 2 * sum(per["gate_up"]) + sum(per["down"])
    total = 32 * layer
    macs = 32 * (4 * 2048 * 4096 * 4096 + 3 * 2048 * 4096 * 11008)
    print(json.dumps({"impl": "reference-table", "config": "stack_7B_32_layers", "seconds": total,
                      "equivalent_tokens_per_s": 2048 / total, "tmacs": macs / total / 1e12,
                      "extrapolated": True, "from": "q_proj x 4 + gate_up x 2 + down, x 32 layers",
                      "cores": cores}), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.oracle_table:
        return run_oracle_table(args)
    M, K, N = WORKLOADS[args.workload]
    from q4_q8_int8_gb300 import synthetic
    x, blk, _ = synthetic.config_inputs(args.workload)
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    # each step: quantize + GEMM over a bounded row sample, sized from a probe
    # so that the whole run (warm-up and timed steps) takes about two minutes
    per_step_budget = args.ref_seconds / max(1, args.steps + args.warmup)
    _, m, dt_probe, _ = cpu_oracle_sample(M, K, N, min(per_step_budget, 2.0), x, blk)
    m = max(1, min(M, int(m * per_step_budget / max(dt_probe, 1e-6))))
    xs = x[:m]
    for _ in range(args.warmup):
        q, da, sa = oracle.quantize_q8_1(xs)
        oracle.gemm(q, da, sa, blk, N, want_bound=False)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        q, da, sa = oracle.quantize_q8_1(xs)
        oracle.gemm(q, da, sa, blk, N, want_bound=False)
    dt = time.perf_counter() - t0
    value = m * N * K * args.steps / dt / 1e12
    sample = f"first {m} of {M} token rows of {args.workload} (K={K}, N={N}) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{args.workload} M={M} K={K} N={N}"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU leg
def path_code(mmq, name):
    """The mmq_q4K_gemm_path code of a path name; SB for the super-block GEMM,
    which has its own entry point."""
    return {"auto": mmq.MMQ_PATH_AUTO, "mma_s8": mmq.MMQ_PATH_MMA_S8, "tc": mmq.MMQ_PATH_TC,
            "small_m": mmq.MMQ_PATH_SMALL_M, SB: SB}[name]


def resolved_path(mmq, path, M):
    """The kernel family mmq_q4K_gemm runs for `path` at M tokens."""
    if path == SB:
        return SB
    if path == mmq.MMQ_PATH_AUTO:
        return mmq.MMQ_PATH_SMALL_M if M <= mmq.SMALL_M_MAX else mmq.MMQ_PATH_TC
    return path


def roofline_seconds(M, K, N, peaks, burst=True):
    """(t_roof, bound): the larger of the algorithmic HBM bytes at the measured
    copy bandwidth and the contraction's f16 tensor flops at the measured bf16
    (= f16) peak."""
    alg_bytes = 0.5625 * N * K + 1.25 * M * K + 4 * M * N
    t_hbm = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    tpk = peaks["bf16_tflops"] if burst else (peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"])
    t_tc = 2.0 * M * N * K / (tpk * 1e12)
    return (t_hbm, "hbm") if t_hbm >= t_tc else (t_tc, "tensor")


def graph_time_ms(fn, reps, dev):
    """Mean device ms of fn(i) for i < reps, replayed from a CUDA graph after a
    warm-up replay (no host launch cost inside the measurement)."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(reps):
                fn(i, s)
    torch.cuda.synchronize(dev)
    g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(dev)
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def sweep_shapes():
    """(label, M, K, N): the FFN GEMMs at 2K tokens, the token-count sweep on
    4096 x 4096, and few-token decode shapes of the 7B layer."""
    from q4_q8_int8_gb300 import synthetic
    out = [(name, *synthetic.SHAPES[name]) for name in ("gate_up", "down")]
    out += [(f"sweep_M{m}", m, 4096, 4096) for m in synthetic.SWEEP_M]
    out += [("decode_M1_4096x11008", 1, 4096, 11008), ("decode_M1_11008x4096", 1, 11008, 4096),
            ("decode_M1_4096x12288", 1, 4096, 12288), ("decode_M4_4096x4096", 4, 4096, 4096),
            ("decode_M16_4096x11008", 16, 4096, 11008)]
    return out


def run_sweep(mmq, dev, peaks, path_name):
    """Kernel-only GEMM time per shape, graph-replayed over rotating inputs
    whose sets together exceed twice the L2."""
    import ctypes
    import torch
    from q4_q8_int8_gb300 import synthetic
    res = {}
    for label, M, K, N in sweep_shapes():
        path = path_code(mmq, path_name)
        if path == mmq.MMQ_PATH_SMALL_M and M > mmq.SMALL_M_MAX:
            continue
        # the super-block GEMM reads the operand plane (4 B per activation) instead of the int8 quants
        set_bytes = 0.5625 * N * K + (4.0 if path == SB else 1.25) * M * K + 4 * M * N
        R = min(64, max(2, int(np.ceil(2 * L2_BYTES / set_bytes)) + 1))
        ws = [synthetic.torch_q4K_weights(N, K, 9100 + r, dev).view(-1) for r in range(R)]
        xs_ = [synthetic.torch_activations(M, K, 9200 + r, dev, 0.01) for r in range(R)]
        if path == SB:
            pre = [mmq.quantize_q8_1_tcop(x) for x in xs_]
            tcops = [t for _, t in pre]
            aqs = [aq for aq, _ in pre]
        else:
            aqs = [mmq.quantize_q8_1(x) for x in xs_]
        del xs_
        Cs = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(R)]
        structs = [mmq.q8_1_struct(*aq) for aq in aqs]

        def call(i, stream):
            r = i % R
            if path == SB:
                rc = mmq.mmq_q4K_gemm_tcop(ctypes.c_void_p(tcops[r].data_ptr()), ctypes.c_void_p(ws[r].data_ptr()),
                                           ctypes.c_void_p(Cs[r].data_ptr()), M, N, K, mmq._stream_ptr(stream))
            else:
                rc = mmq.mmq_q4K_gemm_path(structs[r], ctypes.c_void_p(ws[r].data_ptr()),
                                           ctypes.c_void_p(Cs[r].data_ptr()), M, N, K, path, mmq._stream_ptr(stream))
            if rc:
                raise mmq.MMQError(rc, "mmq_q4K_gemm_path")

        reps = int(max(2 * R, min(400, 20e-3 / max(set_bytes / 6e12, 2e-6))))
        ms = graph_time_ms(call, reps, dev)
        if mmq.status() != 0:
            raise RuntimeError(f"device status error in sweep {label}")
        t_roof, bound = roofline_seconds(M, K, N, peaks)
        macs = M * N * K
        res[label] = {"M": M, "K": K, "N": N, "us": ms * 1e3, "tmacs": macs / (ms * 1e-3) / 1e12,
                      "us_per_gmac": ms * 1e3 / (macs / 1e9),
                      "gbs": set_bytes / (ms * 1e-3) / 1e9, "bound": bound,
                      "t_roof_us": t_roof * 1e6, "roof_frac": t_roof / (ms * 1e-3),
                      "kernels_per_call": 1 if path == SB else mmq.mmq_q4K_gemm_launches(M, N, K, path),
                      "rotating_sets": R, "reps": reps}
        del ws, aqs, Cs, structs
        if path == SB:
            del pre, tcops
        torch.cuda.empty_cache()
    return res


def run_sweep_q6k(mmq, dev, peaks):
    """Kernel-only q6_K GEMM times (mmq_q6K_gemm, the automatic kernel: dp4a up
    to 16 tokens, tcgen05 above), graph-replayed over rotating inputs."""
    import ctypes
    import torch
    from q4_q8_int8_gb300 import synthetic
    res = {}
    for label, M, K, N in (("q6k_M1", 1, 4096, 4096), ("q6k_M1_11008x4096", 1, 11008, 4096),
                           ("q6k_M16_4096x11008", 16, 4096, 11008), ("q6k_M128", 128, 4096, 4096),
                           ("q6k_q_proj", 2048, 4096, 4096), ("q6k_down", 2048, 11008, 4096)):
        wbytes = 210.0 / 256.0 * N * K
        set_bytes = wbytes + 1.25 * M * K + 4 * M * N
        R = min(64, max(2, int(np.ceil(2 * L2_BYTES / set_bytes)) + 1))
        ws = []
        for r in range(R):
            g = torch.Generator(device=dev)
            g.manual_seed(9700 + r)
            raw = torch.randint(0, 256, (N, K // 256, 210), dtype=torch.uint8, device=dev, generator=g)
            raw[:, :, 208] = 0x00
            raw[:, :, 209] = 0x1c   # d = 2^-8 (fp16 0x1c00)
            ws.append(mmq.repack_q6K(raw.view(-1), N, K))
            del raw
        aqs = [mmq.quantize_q8_1(synthetic.torch_activations(M, K, 9800 + r, dev, 0.01)) for r in range(R)]
        Cs = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(R)]
        structs = [mmq.q8_1_struct(*aq) for aq in aqs]

        def call(i, stream):
            r = i % R
            rc = mmq.mmq_q6K_gemm(structs[r], ctypes.c_void_p(ws[r].data_ptr()), ctypes.c_void_p(Cs[r].data_ptr()),
                                  M, N, K, mmq._stream_ptr(stream))
            if rc:
                raise mmq.MMQError(rc, "mmq_q6K_gemm")

        reps = int(max(2 * R, min(400, 20e-3 / max(set_bytes / 6e12, 2e-6))))
        ms = graph_time_ms(call, reps, dev)
        if mmq.status() != 0:
            raise RuntimeError(f"device status error in sweep {label}")
        t_hbm = set_bytes / (peaks["hbm_gbs"] * 1e9)
        t_tc = 2.0 * M * N * K / (peaks["bf16_tflops"] * 1e12)
        macs = M * N * K
        res[label] = {"M": M, "K": K, "N": N, "us": ms * 1e3, "tmacs": macs / (ms * 1e-3) / 1e12,
                      "bound": "hbm" if t_hbm >= t_tc else "tensor", "t_roof_us": max(t_hbm, t_tc) * 1e6,
                      "roof_frac": max(t_hbm, t_tc) / (ms * 1e-3),
                      "kernels_per_call": mmq.mmq_q6K_gemm_launches(M, N, K, mmq.MMQ_PATH_AUTO),
                      "rotating_sets": R, "reps": reps}
        del ws, aqs, Cs, structs
        torch.cuda.empty_cache()
    return res


def run_stack(mmq, dev, path_name, passes=2):
    """The 7B prefill linear stack: 32 layers x {q, k, v, o 4096->4096; gate,
    up 4096->11008; down 11008->4096} at 2048 tokens, every GEMM with its own
    seeded q4_K weights (3.64 GB resident) and a q8_1 prepass of its own
    activations (eight seeded sets per input width, used in turn)."""
    import ctypes
    import torch
    from q4_q8_int8_gb300 import synthetic
    T = synthetic.STACK_TOKENS
    path = path_code(mmq, path_name)
    weights = []
    for layer in range(synthetic.STACK_LAYERS):
        for g, (_, K, N) in enumerate(synthetic.STACK_GEMMS):
            ws, _ = synthetic.stack_seeds(layer, g)
            weights.append((K, N, synthetic.torch_q4K_weights(N, K, ws, dev).view(-1)))
    xs = {K: [synthetic.torch_activations(T, K, 9300 + K + r, dev, 0.01) for r in range(8)] for K in (4096, 11008)}
    q8 = {K: mmq.empty_q8_1(T, K, dev) for K in (4096, 11008)}
    tcop = {K: mmq.empty_tcop(T, K, dev) for K in (4096, 11008)} if path == SB else None
    C = torch.empty((T, 11008), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = mmq._stream_ptr(stream)

    def one_pass():
        for i, (K, N, w) in enumerate(weights):
            x = xs[K][i % 8]
            aq = mmq.q8_1_struct(*q8[K])
            if path == SB:
                tp = ctypes.c_void_p(tcop[K].data_ptr())
                rc = mmq.mmq_quantize_q8_1_tcop(ctypes.c_void_p(x.data_ptr()), T, K, aq, tp, sp)
                rc |= mmq.mmq_q4K_gemm_tcop(tp, ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(C.data_ptr()),
                                            T, N, K, sp)
            else:
                rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(x.data_ptr()), T, K, aq, sp)
                rc |= mmq.mmq_q4K_gemm_path(aq, ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(C.data_ptr()),
                                            T, N, K, path, sp)
            if rc:
                raise RuntimeError(f"stack call failed: {rc}")

    one_pass()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(passes):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one_pass()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    if mmq.status(stream) != 0:
        raise RuntimeError("device status error in the stack")
    ms = float(np.median(times))
    macs = synthetic.STACK_LAYERS * sum(T * K * N for _, K, N in synthetic.STACK_GEMMS)
    out = {"ms_per_pass": ms, "passes": passes, "equivalent_tokens_per_s": T / (ms * 1e-3),
           "tmacs": macs / (ms * 1e-3) / 1e12, "gemms": len(weights),
           "weights_gb": sum(w.numel() for _, _, w in weights) / 1e9,
           "what": "32 layers x (q, k, v, o, gate, up, down) at 2048 tokens, a q8_1 prepass per GEMM, "
                   "224 independent weight matrices resident"}
    del weights, xs, q8, tcop, C
    torch.cuda.empty_cache()
    return out


def run_mine(args, rank, world, local_rank):
    import torch
    import q4_q8_int8_gb300 as mmq
    from q4_q8_int8_gb300 import build as mmq_build, synthetic

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    mmq_build.build()
    mmq.load_library()
    mmq.mmq_set_programmatic_launch(0 if args.no_pdl else 1)
    path = path_code(mmq, args.path)

    M, K, N = WORKLOADS[args.workload]
    # Inputs: R independent sets rotated step by step so that every step reads
    # its inputs from HBM (R sets together exceed twice the 129 MB L2).
    sb = path == SB
    plane = 4.0 * M * K if sb else 0.0   # the super-block path's operand plane (written, then read)
    set_bytes = M * K * 4 + M * K * 1.25 + plane + N * K * 0.5625 + M * N * 4
    R = max(2, int(np.ceil(2 * L2_BYTES / set_bytes)) + 1)
    xs, ws, aqs, Cs, tcops = [], [], [], [], []
    for r in range(R):
        xs.append(synthetic.torch_activations(M, K, 7000 + 97 * rank + r, dev, 0.01))
        ws.append(synthetic.torch_q4K_weights(N, K, 8000 + 97 * rank + r, dev).view(-1))
        aqs.append(mmq.empty_q8_1(M, K, dev))
        Cs.append(torch.empty((M, N), dtype=torch.float32, device=dev))
        if sb:
            tcops.append(mmq.empty_tcop(M, K, dev))
    stream = torch.cuda.current_stream(dev)
    sp = mmq._stream_ptr(stream)
    import ctypes

    def step(i, evs=None):
        r = i % R
        x, w, (qs, da, sa), C = xs[r], ws[r], aqs[r], Cs[r]
        aq = mmq.q8_1_struct(qs, da, sa)
        if evs is not None:
            evs[0].record(stream)
        if sb:
            tp = ctypes.c_void_p(tcops[r].data_ptr())
            rc = mmq.mmq_quantize_q8_1_tcop(ctypes.c_void_p(x.data_ptr()), M, K, aq, tp, sp)
        else:
            rc = mmq.mmq_quantize_q8_1(ctypes.c_void_p(x.data_ptr()), M, K, aq, sp)
        if evs is not None:
            evs[1].record(stream)
        if sb:
            rc |= mmq.mmq_q4K_gemm_tcop(tp, ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(C.data_ptr()),
                                        M, N, K, sp)
        else:
            rc |= mmq.mmq_q4K_gemm_path(aq, ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(C.data_ptr()),
                                        M, N, K, path, sp)
        if evs is not None:
            evs[2].record(stream)
        if rc:
            raise RuntimeError(f"MMQ call failed: {rc}")

    # clocks are sampled from the start of warm-up to the end of the soak below
    pci = None
    try:
        pr = torch.cuda.get_device_properties(dev)
        pci = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
    except AttributeError:
        pass
    clocks = ClockSampler(local_rank, pci) if rank == 0 else None
    if clocks:
        clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    if mmq.status(stream) != 0:
        raise RuntimeError("device status error after warm-up")
    # The timed region: K steps with events only at its two ends.  An event
    # recorded between two kernels keeps the second from starting early
    # (programmatic launch), which costs about 11 us per step here, so the
    # per-kernel split is taken in a second pass of the same K steps with
    # events around each kernel, right after the timed region.
    ev_t0, ev_t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    ev_t0.record(stream)
    for i in range(args.steps):
        step(args.warmup + i)
    ev_t1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    # Event records cost the host far more than a launch (about 25 us each
    # on the Grace host); a spin of torch's on the stream first lets the host
    # queue the pass ahead, so that no kernel waits for the host.
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(min(args.steps, 1000) * 2e5))   # ~0.1 ms of spin per step at 2 GHz
    for i in range(args.steps):
        step(args.warmup + args.steps + i, evs[i])
    torch.cuda.synchronize(dev)
    step_ms = ev_t0.elapsed_time(ev_t1) / args.steps
    # A third pass, outside the timed region: the same K steps' GEMMs alone,
    # launched back to back as in the timed region (events only at the ends).
    # Its time per call is the GEMM's share of an overlapped step; the step
    # minus it is what the prepass adds to the step.
    ev_g0, ev_g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_g0.record(stream)
    for i in range(args.steps):
        r = (args.warmup + i) % R
        w_, (qs_, da_, sa_), C_ = ws[r], aqs[r], Cs[r]
        aq_ = mmq.q8_1_struct(qs_, da_, sa_)
        if sb:
            rc_ = mmq.mmq_q4K_gemm_tcop(ctypes.c_void_p(tcops[r].data_ptr()), ctypes.c_void_p(w_.data_ptr()),
                                        ctypes.c_void_p(C_.data_ptr()), M, N, K, sp)
        else:
            rc_ = mmq.mmq_q4K_gemm_path(aq_, ctypes.c_void_p(w_.data_ptr()), ctypes.c_void_p(C_.data_ptr()),
                                        M, N, K, path, sp)
        if rc_:
            raise RuntimeError(f"MMQ call failed: {rc_}")
    ev_g1.record(stream)
    torch.cuda.synchronize(dev)
    gemm_loop_ms = ev_g0.elapsed_time(ev_g1) / args.steps
    # Soak: the same step loop for about --soak-seconds more, so that the
    # clock record holds many samples taken under load (the timed region of
    # a default run is only a few milliseconds).
    soak_steps = int(args.soak_seconds / max(step_ms * 1e-3, 1e-6)) if clocks else 0
    ts0 = time.perf_counter()
    for i in range(soak_steps):
        step(i)
        if i % 256 == 255:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    soak_s = time.perf_counter() - ts0
    clk = clocks.stop() if clocks else None
    rc = mmq.status(stream)
    if rc != 0:
        raise RuntimeError(f"device status {rc} after timed region")

    split_step_ms = evs[0][0].elapsed_time(evs[-1][2]) / args.steps
    q_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    g_all = np.array([e[1].elapsed_time(e[2]) for e in evs])
    g_ms = float(np.mean(g_all))
    g_dist = {"median": float(np.median(g_all)), "min": float(g_all.min()), "max": float(g_all.max())}
    step_ms, split_step_ms, q_ms, g_ms, gemm_loop_ms = max_over_ranks(
        [step_ms, split_step_ms, q_ms, g_ms, gemm_loop_ms], world, dev)

    # ---- end to end through the C ABI with pinned host buffers: mmq_q4K_gemm_host
    # (x in from host memory, C out to host memory, chunked so that the copies
    # overlap the prepass and GEMM)
    xh = torch.empty((M, K), dtype=torch.float32, pin_memory=True)
    xh.copy_(xs[0].cpu())
    Ch = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    ws_bytes = mmq.mmq_q4K_gemm_host_workspace(M, N, K)
    ws_t = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=dev)
    ws_base = (ws_t.data_ptr() + 255) // 256 * 256

    def e2e_step(i):
        w = ws[i % R]
        rc = mmq.mmq_q4K_gemm_host(ctypes.c_void_p(xh.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                   ctypes.c_void_p(Ch.data_ptr()), M, N, K, ctypes.c_void_p(ws_base),
                                   ws_bytes, sp)
        if rc:
            raise RuntimeError(f"MMQ call failed: {rc}")

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    eb.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = ea.elapsed_time(eb) / e2e_steps
    e2e_ms = max_over_ranks([e2e_ms], world, dev)[0]

    # ---- the dequantize-then-dense control path on the same inputs (rank 0)
    control = None
    if rank == 0 and not args.no_control:
        xh16 = [torch.empty((M, K), dtype=torch.float16, device=dev) for _ in range(R)]
        wh16 = [torch.empty((N, K), dtype=torch.float16, device=dev) for _ in range(R)]

        def ctrl_step(i, ev=None):
            r = i % R
            if ev is not None:
                ev[0].record(stream)
            mmq.convert_f16(xs[r], out=xh16[r], stream=stream)
            if ev is not None:
                ev[1].record(stream)
            mmq.dequantize_q4K_f16(ws[r], N, K, out=wh16[r], stream=stream)
            if ev is not None:
                ev[2].record(stream)
            mmq.gemm_f16(xh16[r], wh16[r], out=Cs[r], stream=stream)
            if ev is not None:
                ev[3].record(stream)

        for i in range(3):
            ctrl_step(i)
        torch.cuda.synchronize(dev)
        cn = max(3, min(args.steps, 20))
        cev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(cn)]
        for i in range(cn):
            ctrl_step(3 + i, cev[i])
        torch.cuda.synchronize(dev)
        if mmq.status(stream) != 0:
            raise RuntimeError("device status error in the control path")
        c_conv = float(np.mean([e[0].elapsed_time(e[1]) for e in cev]))
        c_deq = float(np.mean([e[1].elapsed_time(e[2]) for e in cev]))
        c_gemm = float(np.mean([e[2].elapsed_time(e[3]) for e in cev]))
        pk = measured_peaks()
        control = {
            "what": "x -> fp16, q4_K -> fp16 (dequantize), dense tcgen05 fp16 GEMM with f32 accumulation",
            "convert_ms": c_conv, "dequant_ms": c_deq, "gemm_f16_ms": c_gemm,
            "total_ms": c_conv + c_deq + c_gemm,
            "gemm_f16_tflops": 2.0 * M * N * K / (c_gemm * 1e-3) / 1e12,
            "gemm_f16_frac_of_burst": 2.0 * M * N * K / (c_gemm * 1e-3) / 1e12 / pk["bf16_tflops"],
            "dequant_gbs": N * K * (0.5625 + 2) / (c_deq * 1e-3) / 1e9,
            "convert_gbs": M * K * 6 / (c_conv * 1e-3) / 1e9,
            "mmq_step_over_control": step_ms / (c_conv + c_deq + c_gemm),
            "gpu_launches": 3 * cn,
        }
        del xh16, wh16

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peaks = measured_peaks()
    sweep = None
    stack = None
    if not args.no_sweep or not args.no_stack:
        del xs, ws, aqs, Cs, ws_t, tcops
        torch.cuda.empty_cache()
    sweep_q6k = None
    if not args.no_sweep:
        sweep = run_sweep(mmq, dev, peaks, args.path)
        sweep_q6k = run_sweep_q6k(mmq, dev, peaks)
    if not args.no_stack:
        stack = run_stack(mmq, dev, args.path)

    macs = M * N * K
    value = whole_job_tmacs(macs, world, step_ms)
    gemm_tmacs = macs / (g_ms * 1e-3) / 1e12
    micro = microbench_peaks()
    used_path = resolved_path(mmq, path, M)
    kname = {mmq.MMQ_PATH_MMA_S8: ("gemm_mma_s8", "gemm_mma.cu"),
             mmq.MMQ_PATH_TC: ("gemm_tc", "gemm_tc.cu"),
             mmq.MMQ_PATH_SMALL_M: ("gemm_small_m", "gemm_small.cu"),
             SB: ("gemm_sb", "gemm_sb.cu")}[used_path]
    src_hash = kernel_source_hash([kname[1], "sm103_ptx.cuh", "tc_common.cuh", "q8_round.cuh"])
    traffic = recorded_traffic(kname[0], src_hash)
    alg_bytes = 0.5625 * N * K + 1.25 * M * K + 4 * M * N
    sm_mhz = (clk or {}).get("sm_mhz") or micro["sm_max_mhz"]
    timed_s = step_ms * 1e-3 * args.steps
    burst = timed_s < SUSTAINED_AFTER_S
    if used_path == mmq.MMQ_PATH_SMALL_M:
        achieved = alg_bytes / (g_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm copy)"}
    elif used_path in (mmq.MMQ_PATH_TC, SB):
        # The exact integer contraction runs on the tensor pipe as kind::f16
        # MMAs (2 flops per MAC).  A timed region of milliseconds is held to
        # the burst bf16 (= f16 rate) peak; the sustained fraction is beside it.
        flops = 2.0 * macs
        achieved = flops / (g_ms * 1e-3) / 1e12
        sus = peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"]
        peak = peaks["bf16_tflops"] if burst else sus
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json bf16 "
                               f"{'burst' if burst else 'sustained'}; f16 runs at the bf16 rate; "
                               f"timed region {timed_s * 1e3:.1f} ms)",
                "frac_of_sustained": achieved / sus, "frac_of_burst": achieved / peaks["bf16_tflops"]}
    else:
        achieved = 2 * macs / (g_ms * 1e-3) / 1e12
        peak = micro["int8_mma_sync_tops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": "measured int8 mma.sync peak (profiles/peaks.json, bench_peaks.cu)"}
    roof["kernel"] = kname[0]
    # One GEMM call may be two kernels (the tcgen05 kernel's split-K tail
    # launch); "per launch" figures here are per call, both kernels together.
    gemm_launches = 1 if used_path == SB else mmq.mmq_q4K_gemm_launches(M, N, K, used_path)
    if gemm_launches < 1:
        raise RuntimeError(f"mmq_q4K_gemm_launches failed: {gemm_launches}")
    roof["kernels_per_call"] = gemm_launches
    # The epilogue's FP32 ceiling, reported beside the tensor roofline: per
    # output and 32-k chunk the tcgen05 kernel does one FMA (2 flops), plus
    # per super-block one FMA for d and one add of the second term (0.5 flop
    # per chunk); the other kernels do the pages' 1 FMUL + 2 FFMA (5 flops).
    # (the super-block kernel: per output and super-block a multiply, an FMA
    # and the second term's FMA: 6 flops per 256 k, under 0.75 per chunk)
    alu_flops = {mmq.MMQ_PATH_TC: 2.5, SB: 0.75}.get(used_path, 5.0) * macs / 32
    alu_peak = micro["sms"] * 128 * 2 * sm_mhz * 1e6 / 1e12
    alu = {"flops_per_launch": alu_flops, "achieved_tflops": alu_flops / (g_ms * 1e-3) / 1e12,
           "peak_tflops": alu_peak, "frac": alu_flops / (g_ms * 1e-3) / 1e12 / alu_peak,
           "peak_source": f"derived: {micro['sms']} SMs x 128 FP32 lanes x 2 x {sm_mhz:.0f} MHz"}
    roof["algorithmic_bytes_per_launch"] = alg_bytes
    roof["algorithmic_macs_per_launch"] = macs

    cpu = None
    if not args.no_cpu_baseline:
        from q4_q8_int8_gb300 import synthetic as syn
        x0, blk0, _ = syn.config_inputs(args.workload)
        v, m, secs, cores = cpu_oracle_sample(M, K, N, args.cpu_seconds, x0, blk0)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"first {m} of {M} token rows of {args.workload}, quantize + blockwise "
                         f"GEMM, {secs:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {mmq.MMQ_PATH_TC: "int8xu4->f32 (fp16-exact ints on tensor cores)",
                  SB: "fp16 hi+lo activations x fp16-exact sc*v -> f32 (tensor cores)"}.get(
                      used_path, "s8xs8->s32, f32 rescale"),
        "data": "synthetic",
        "config": {"workload": f"{args.workload} M={M} K={K} N={N}", "global_batch_tokens": M * world,
                   "parallelism": f"independent problem per GPU x{world}",
                   "l2": f"{R} rotating input sets ({R * set_bytes / 1e6:.0f} MB > 2x L2)",
                   "path": args.path, "programmatic_launch": not args.no_pdl},
        "us_per_gmac": step_ms * 1e3 / (macs / 1e9),
        "gemm_only": {"tmacs": gemm_tmacs, "us_per_gmac": g_ms * 1e3 / (macs / 1e9), "ms": g_ms,
                      "ms_over_steps": g_dist,
                      "x_int8_mma_sync_rate": 2 * gemm_tmacs / micro["int8_mma_sync_tops"],
                      "int8_note": "a multiple of the measured legacy mma.sync s8 rate "
                                   f"({micro['int8_mma_sync_tops']} TOP/s, bench_peaks.cu); sm_103a has "
                                   "no tcgen05 integer MMA, and this kernel runs on the f16 tensor pipe, "
                                   "so the roofline fraction is the one in 'roofline'"},
        "epilogue_alu": alu,
        "prepass": {"ms": q_ms, "gbs": (M * K * 5.25 + plane) / (q_ms * 1e-3) / 1e9,
                    "frac_of_hbm": (M * K * 5.25 + plane) / (q_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                    "bytes": M * K * 5.25 + plane,
                    "ms_added_to_step": step_ms - gemm_loop_ms,
                    "gbs_added_to_step": (M * K * 5.25 + plane) / max((step_ms - gemm_loop_ms) * 1e-3, 1e-9) / 1e9,
                    "what": "ms: between events around the kernel (split pass); ms_added_to_step: the timed "
                            "step minus the same GEMMs launched back to back without prepasses (gemm_loop_ms)"},
        "gemm_loop_ms": gemm_loop_ms,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_tmacs(macs, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": M * K * 4, "d2h_bytes_per_step": M * N * 4,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * (1 + gemm_launches),
        "control": control,
        "clocks": clk,
        "clocks_window": f"from warm-up start through the timed region, the per-kernel split pass and "
                         f"a {soak_s:.2f} s soak of {soak_steps} more steps of the same loop",
        "split_pass": {"ms_per_step": split_step_ms,
                       "what": "the same K steps again with an event before and after each kernel; "
                               "prepass, gemm_only and roofline come from this pass"},
        "wall_s_timed": wall,
        "sweep": sweep,
        "sweep_note": "kernel-only GEMM per configuration (outside the timed region), CUDA-graph replay over "
                      "rotating inputs > 2x L2; roof_frac = t_roof / t with t_roof = max(algorithmic bytes / "
                      "measured HBM, 2MNK / measured burst bf16)",
        "stack": stack,
        "sweep_q6k": sweep_q6k,
        "sweep_q6k_note": "q6_K weights (the pages' next family): kernel-only mmq_q6K_gemm, graph replay over rotating "
                          "inputs > 2x L2; roof_frac as in sweep with 210 / 256 bytes per weight",
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def measure_peaks():
    """Compile bench_peaks.cu under _build/ and run it (prints one JSON line)."""
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "bench_peaks")
    nvcc = os.environ.get("NVCC", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    os.path.join(ROOT, "bench_peaks.cu")], check=True)
    subprocess.run([exe], check=True)


def run_shape(args):
    """Profiling mode: prepass + GEMM of one seeded shape, --launches times,
    then the device status (a command line for ncu -k ... -s ... -c ...)."""
    import ctypes
    import torch
    import q4_q8_int8_gb300 as mmq
    from q4_q8_int8_gb300 import build as mmq_build, synthetic
    M, K, N = (int(v) for v in args.shape.split(":"))
    dev = torch.device("cuda", 0)
    mmq_build.build()
    mmq.load_library()
    mmq.mmq_set_programmatic_launch(0 if args.no_pdl else 1)
    x = synthetic.torch_activations(M, K, 9500, dev, 0.01)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    sp = mmq._stream_ptr()
    if args.weights == "q6k":
        g = torch.Generator(device=dev)
        g.manual_seed(9600)
        raw = torch.randint(0, 256, (N, K // 256, 210), dtype=torch.uint8, device=dev, generator=g)
        raw[:, :, 208] = 0x00
        raw[:, :, 209] = 0x1c   # d = 2^-8 (fp16 0x1c00)
        w = mmq.repack_q6K(raw.view(-1), N, K)
        path = path_code(mmq, args.path if args.path != SB else "auto")
        gemm = lambda aq: mmq.mmq_q6K_gemm_path(mmq.q8_1_struct(*aq), ctypes.c_void_p(w.data_ptr()),
                                                ctypes.c_void_p(C.data_ptr()), M, N, K, path, sp)
        prep = lambda: (mmq.quantize_q8_1(x), None)
    else:
        w = synthetic.torch_q4K_weights(N, K, 9600, dev).view(-1)
        path = path_code(mmq, args.path)
        if path == SB:
            prep = lambda: mmq.quantize_q8_1_tcop(x)
            gemm = lambda aq, t=None: mmq.mmq_q4K_gemm_tcop(ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(w.data_ptr()),
                                                            ctypes.c_void_p(C.data_ptr()), M, N, K, sp)
        else:
            prep = lambda: (mmq.quantize_q8_1(x), None)
            gemm = lambda aq, t=None: mmq.mmq_q4K_gemm_path(mmq.q8_1_struct(*aq), ctypes.c_void_p(w.data_ptr()),
                                                            ctypes.c_void_p(C.data_ptr()), M, N, K, path, sp)
    for _ in range(args.launches):
        aq, t = prep()
        rc = gemm(aq) if args.weights == "q6k" else gemm(aq, t)
        if rc:
            raise RuntimeError(f"GEMM call failed: {rc}")
    torch.cuda.synchronize()
    st = mmq.status()
    print(json.dumps({"shape": args.shape, "weights": args.weights, "path": args.path, "launches": args.launches,
                      "status": st}), flush=True)
    if st != 0:
        raise SystemExit(1)


def main():
    args = parse()
    if args.measure_peaks:
        return measure_peaks()
    if args.shape:
        return run_shape(args)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_mine(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
