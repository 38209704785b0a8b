#!/usr/bin/env python
"""Benchmark of the W4A4 NVFP4 fused projection (one JSON line on rank 0).

Default workload: the video diffusion-transformer block (M = 16384 tokens; QKV
1536 -> 4608, o 1536 -> 1536, FFN up 1536 -> 8960 and down 8960 -> 1536; rank-32
low-rank branch; the 64 highest-energy channels kept in fp16; block-64 FWHT;
smoothing), the largest configuration of the workload set, on seeded synthetic
inputs.  A step is one pass of the whole hot path over the batch: for every layer
the fused activation quantiser and the tcgen05 NVFP4 GEMM with its fused epilogue
(two kernels per layer), replayed as one CUDA graph.  L2 is flushed (a 256 MiB
write) before every timed step, outside the step's CUDA events, so weights and
activations come from HBM.  Other workloads: --workload expert | backbone |
vae_conv | tiny.  --mma-peak prints the tensor-core issue-rate table instead.

--impl reference times the CPU oracle (the slow, plain reference implementation)
on the same workload, a bounded row sample per step, on the host cores.
Multi-GPU (torchrun): every rank runs an independent replica of the workload on its
own GPU (weak scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A4 NVFP4 fused-projection TFLOPS & tokens/s; % of FP4/HBM roofline"
FLUSH_BYTES = 256 << 20
WORKLOAD_TEXT = {
    "expert": "action-expert projections, batch 1: M=50 tokens, up 1024->4096 + down 4096->1024, "
              "rank-32 bf16 branch, block-64 FWHT, smoothing, NVFP4 W4A4",
    "video_dit": "video DiT block: M=16384 tokens, QKV 1536->4608, o 1536->1536, up 1536->8960, "
                 "down 8960->1536, rank 32, 64 fp16 outlier channels, NVFP4 W4A4",
    "tiny": "single projection M=8, K=256 -> N=512, rank 16",
    "vae_conv": "Wan-style VAE Conv3d 3x3x3, C 384->384, input 1x384x5x60x104, padding 1: implicit GEMM "
                "M=31200 voxels, K=10368, N=384, NVFP4 with a per-tensor activation scale",
    "backbone": "language backbone prefill M=768: QKV 2048->6144 and gate/up 2048->32768 in W4A4, "
                "o_proj 2048->2048 and down 16384->2048 in W8A8 (int8 codes held as bf16)",
    "backbone_fp8": "language backbone prefill M=768: QKV 2048->6144 and gate/up 2048->32768 in W4A4, "
                    "o_proj 2048->2048 and down 16384->2048 in FP8 W8A8 (e4m3 codes, kind::f8f6f4)",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None, help="timed steps (default: by workload)")
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["wq", "reference"], default="wq")
    ap.add_argument("--workload", default="video_dit", choices=list(WORKLOAD_TEXT))
    ap.add_argument("--kernel-iters", type=int, default=None)
    ap.add_argument("--mma-peak", action="store_true", help="tensor-core issue-rate table (one JSON line)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-layer", default=None, help="run one named layer of the workload (profiling)")
    a = ap.parse_args()
    # defaults keep the timed region to seconds (a video-DiT step is ~1 ms, an expert step ~30 us)
    d_steps, d_warm, d_iters = {"video_dit": (200, 10, 30), "vae_conv": (200, 10, 50), "backbone": (500, 20, 100),
                                "backbone_fp8": (500, 20, 100), "expert": (2000, 50, 200),
                                "tiny": (2000, 50, 200)}[a.workload]
    a.steps = d_steps if a.steps is None else a.steps
    a.warmup = d_warm if a.warmup is None else a.warmup
    a.kernel_iters = d_iters if a.kernel_iters is None else a.kernel_iters
    return a


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def job_time_ms(local_ms: float, ws: int, device=None) -> float:
    """Time of the whole job: the slowest rank's time for the same number of steps (every rank
    times exactly K steps between barriers).  One rank: its own time."""
    if ws <= 1:
        return float(local_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, ws: int, job_ms: float) -> float:
    """Whole-job units per second: every rank processed `units_per_rank_step` units per step
    (independent replicas, weak scaling), divided by the job time."""
    return units_per_rank_step * steps * ws / (job_ms / 1e3)


def layers_of(name):
    import workloads as wl
    w = wl.WORKLOADS[base_workload(name)]
    return w, list(range(len(w.layers)))


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while the timed region runs."""

    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}

    def __init__(self, dev_index: int):
        self.samples, self.reasons, self.ok = [], set(), False
        self.max_mhz = None
        self.source = "unavailable"
        self.dev_index = dev_index
        self._stop = threading.Event()
        self._proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(dev_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.ok = True
            self.source = "NVML"
        except Exception as exc:
            self.ok = False
            self.source = f"nvidia-smi (NVML python binding failed: {type(exc).__name__})"

    def _run(self):
        if not self.ok:
            return self._run_smi()
        nv = self._nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                    getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
                r = fn(self._h)
                for k, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(k)
            except Exception:
                pass
            time.sleep(0.002)

    def _run_smi(self):
        import subprocess
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self._proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev_index), f"--query-gpu={q}",
                                           "--format=csv,noheader,nounits", "-lms", "20"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.source = "unavailable"
            return
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            f = [x.strip() for x in line.split(",")]
            try:
                self.samples.append(float(f[0]))
                self.max_mhz = float(f[1])
                for n, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(n)
            except (ValueError, IndexError):
                pass

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        if not self.ok:
            time.sleep(0.3)          # let nvidia-smi start sampling before the timed work
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        self._t.join(timeout=5)

    def record(self):
        return {"sm_mhz": float(statistics.median(self.samples)) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": self.source}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


def fp4_peak_tflops(peaks):
    """Dense FP4 tensor peak for the roofline: the measured bf16 burst peak times the nominal
    fp4 : bf16 ratio (13.5 : 2.25 = 6), the rule for a contraction whose own dtype has no
    measured peak."""
    return peaks.get("bf16_tflops", 1800.0) * 6.0


def kernel_roofline(flops, nbytes, ms, peaks):
    """Roofline time of one launch = max(flops / P_fp4, bytes / HBM); bound = the larger term;
    frac = roofline time / measured time."""
    p4 = fp4_peak_tflops(peaks) * 1e12
    hbm = peaks["hbm_gbs"] * 1e9
    t_tensor = flops / p4 if flops else 0.0
    t_hbm = nbytes / hbm
    bound = "tensor" if t_tensor > t_hbm else "hbm"
    t_roof = max(t_tensor, t_hbm)
    return {"bound": bound, "roofline_us": 1e6 * t_roof, "measured_us": 1e3 * ms,
            "frac": t_roof / (ms / 1e3) if ms > 0 else None}


def queued_event_times(fn, iters, stream, flush, chunk=25, sleep_cycles=20_000_000):
    """Device time of `fn`'s launches, each after an L2 flush, with CUDA events on the launching
    stream.  Every chunk of launches is queued behind a device-side sleep, so the GPU never waits
    for the host to enqueue the launch the start event precedes (host enqueue stays out of the
    measured span).  Returns the per-launch times in ms."""
    import torch
    out = []
    for c0 in range(0, iters, chunk):
        n = min(chunk, iters - c0)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            torch.cuda._sleep(sleep_cycles)
            for i in range(n):
                flush.zero_()
                evs[i][0].record(stream)
                fn()
                evs[i][1].record(stream)
        torch.cuda.synchronize()
        out += [a.elapsed_time(b) for a, b in evs]
    return out


def gemm_algorithmic_bytes(M, K, N, r, n_out, bias):
    """Bytes the fused GEMM must move once: fp4 codes + e4m3 scales of A and W, row scales,
    the 16-bit side operands, bias and the bf16 output."""
    a = M * K // 2 + M * K // 16 + 4 * M
    w = N * K // 2 + N * K // 16
    side = 2 * M * r + 2 * N * r + 2 * M * n_out + 2 * N * n_out
    return a + w + side + (4 * N if bias else 0) + 2 * M * N


def gemm8_algorithmic_bytes(M, K, N, bias):
    """8-bit layer: int8 codes of A and W (one byte each), per-row and per-column scales,
    bias, bf16 output."""
    return M * K + 4 * M + N * K + 4 * N + (4 * N if bias else 0) + 2 * M * N


def quant8_algorithmic_bytes(M, K, smooth):
    return 2 * M * K + M * K + 4 * M + (4 * K if smooth else 0)


def quant_algorithmic_bytes(M, K, r, n_out, smooth):
    """Bytes the activation quantiser must move: bf16 x in (2 B/elt); fp4 codes + e4m3 scales
    (0.5625 B/elt) and the fp32 row scale (4 B/row) out; its 16-bit side outputs U and x_O out
    (2 B per value).  The per-layer constants (inv_s, P) are left out."""
    return 2 * M * K + M * K // 2 + M * K // 16 + 4 * M + 2 * M * r + 2 * M * n_out


def kernel_source_hash():
    """Hash of every kernel source file: a stored ncu figure is used only for the code it measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a4_nvfp4_quantized_wq_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload, {}).get(kernel)
        if e and e.get("source_hash") == kernel_source_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def base_workload(name):
    """The workload whose inputs a bench workload uses (backbone_fp8 runs the backbone's 8-bit
    layers in FP8)."""
    return "backbone" if name == "backbone_fp8" else name


def eight_bit_mode(wq, name):
    return wq.WQ_MODE_W8A8_FP8 if name == "backbone_fp8" else wq.WQ_MODE_W8A8


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_layer_data(name):
    import workloads as wl
    w, idx = layers_of(name)
    return [wl.make_layer_inputs(base_workload(name), layer=i) for i in idx]


def oracle_eight_bit(fp8):
    """The oracle's 8-bit layer functions: (prepare, quantise, forward), int8 or e4m3."""
    import oracle
    if fp8:
        return oracle.prepare_weights_fp8, oracle.quantize_act_fp8, oracle.linear_forward_fp8
    return oracle.prepare_weights_int8, oracle.quantize_act_int8, oracle.linear_forward_w8a8


def time_oracle(layers, budget_s: float, n_threads: int, min_passes=1, fp8=False):
    """Time the oracle's per-token work (quantiser, low-rank, forward) on row samples;
    returns (tokens/s, rows per pass, passes, seconds)."""
    import oracle
    prep8, quant8, fwd8 = oracle_eight_bit(fp8)
    prepared = [(L, prep8(L.W, L.s, L.rotate, n_threads) if L.spec.mode == "w8a8" else
                 oracle.prepare_weights(L.W, L.s, L.L1, L.L2, L.omega, L.rotate, n_threads)) for L in layers]

    def one(rows):
        for L, wqo in prepared:
            xb = L.x_bits[rows]
            if L.spec.mode == "w8a8":
                fwd8(quant8(xb, L.s, L.rotate, n_threads), wqo, L.bias, n_threads)
                continue
            aq = oracle.quantize_act(xb, L.s, L.rotate, L.omega, n_threads=n_threads)
            U = oracle.lowrank_act(xb, wqo.P) if wqo.P.shape[1] else None
            oracle.linear_forward(aq, wqo, U, L.bias, n_threads=n_threads)

    M = layers[0].M
    t0 = time.perf_counter()
    one(np.arange(min(M, 8)))
    t_row = (time.perf_counter() - t0) / min(M, 8)
    rows_per_pass = int(max(1, min(M, budget_s / max(t_row, 1e-9) / max(min_passes, 1))))
    rows = np.sort(np.random.default_rng(7).choice(M, size=rows_per_pass, replace=False))
    passes, t0 = 0, time.perf_counter()
    while True:
        one(rows)
        passes += 1
        el = time.perf_counter() - t0
        if passes >= min_passes and el >= budget_s * 0.5:
            break
        if el > budget_s * 3:
            break
    el = time.perf_counter() - t0
    return rows_per_pass * passes / el, rows_per_pass, passes, el


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    n_threads = os.cpu_count() or 1
    layers = oracle_layer_data(args.workload)
    import oracle as orc
    prep8, quant8, fwd8 = oracle_eight_bit(args.workload == "backbone_fp8")
    prepared = [(L, prep8(L.W, L.s, L.rotate, n_threads) if L.spec.mode == "w8a8" else
                 orc.prepare_weights(L.W, L.s, L.L1, L.L2, L.omega, L.rotate, n_threads)) for L in layers]
    M = layers[0].M
    # size each step's row sample so that warmup + steps fit in about a minute
    t0 = time.perf_counter()
    rows = np.arange(min(M, 4))

    def step(rows):
        for L, wqo in prepared:
            xb = L.x_bits[rows]
            if L.spec.mode == "w8a8":
                fwd8(quant8(xb, L.s, L.rotate, n_threads), wqo, L.bias, n_threads)
                continue
            aq = orc.quantize_act(xb, L.s, L.rotate, L.omega, n_threads=n_threads)
            U = orc.lowrank_act(xb, wqo.P) if wqo.P.shape[1] else None
            orc.linear_forward(aq, wqo, U, L.bias, n_threads=n_threads)

    step(rows)
    t_row = (time.perf_counter() - t0) / len(rows)
    per_step = 60.0 / max(1, args.steps + args.warmup)
    n_rows = int(max(1, min(M, per_step / max(t_row, 1e-9))))
    rng = np.random.default_rng(11)
    for _ in range(args.warmup):
        step(np.sort(rng.choice(M, n_rows, replace=False)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(np.sort(rng.choice(M, n_rows, replace=False)))
    el = time.perf_counter() - t0
    tok_s = n_rows * args.steps / el
    flops = sum(2.0 * n_rows * L.spec.K * L.spec.N for L in layers) * args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "tflops": flops / el / 1e12,
        "config": {"workload": WORKLOAD_TEXT[args.workload], "M": M, "rows_per_step": n_rows},
        "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": n_threads, "kind": "oracle",
                         "sample": f"{n_rows} of {M} rows per step, all layers, {args.steps} steps"},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def run_wq(args):
    import torch
    ws, rank, local_rank = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from w4a4_nvfp4_quantized_wq_b300 import build as wqbuild
    wqbuild.build_library()
    import w4a4_nvfp4_quantized_wq_b300 as wq
    import workloads as wl

    wlw, idx = layers_of(args.workload)
    if args.only_layer:
        idx = [i for i in idx if wlw.layers[i].name == args.only_layer]
    layers = [wl.make_layer_inputs(base_workload(args.workload), layer=i) for i in idx]
    M = wlw.M
    stream = torch.cuda.Stream(device=dev)
    H = []
    for L in layers:
        if L.spec.mode == "w8a8":
            w = wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, rotate=L.rotate,
                                      mode=eight_bit_mode(wq, args.workload))
        else:
            w = wq.wq_prepare_weights(L.spec.K, L.spec.N, L.W, L.bias, L.s, L.L1, L.L2,
                                      L.omega if L.omega.size else None, rotate=L.rotate)
        x = torch.from_numpy(L.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        y = torch.empty((M, L.spec.N), dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(max(256, wq.wq_workspace_bytes(w, M)), dtype=torch.uint8, device=dev)
        H.append(dict(L=L, w=w, x=x, y=y, ws=wsb))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        for h in H:
            if h["L"].spec.mode == "w8a8":
                wq.wq_linear_forward_w8a8(h["w"], h["x"], h["y"], h["ws"], stream)
            else:
                wq.wq_linear_forward(h["w"], h["x"], h["y"], h["ws"], stream)

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    for h in H:
        wq.wq_check_device_error(h["w"])

    # kernels this library launches per step: one per layer on the fused path, else two
    launches_per_step = sum(1 if (h["L"].spec.mode != "w8a8" and wq.wq_forward_path(h["w"], M) == wq.WQ_PATH_FUSED)
                            else 2 for h in H)

    # ---------------- timed region: exactly K steps
    K, W = args.steps, args.warmup
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for _ in range(W):
            flush.zero_()
            graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with sampler:
        with torch.cuda.stream(stream):
            for i in range(K):
                flush.zero_()
                ev[i][0].record(stream)
                graph.replay()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = job_time_ms(float(sum(step_ms)), ws, dev)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    for h in H:
        wq.wq_check_device_error(h["w"])
    tok_s = job_throughput(M, K, ws, total_ms)
    flops_step = sum(2.0 * M * h["L"].spec.K * h["L"].spec.N for h in H)
    tflops = flops_step * K * ws / (total_ms / 1e3) / 1e12

    # ---------------- per-kernel timing and roofline (each launch alone, L2 flushed before it)
    import ctypes
    peaks, peak_kind = measured_peaks()
    iters = args.kernel_iters
    per_kernel = []
    for li, h in enumerate(H):
        L, w = h["L"], h["w"]
        w8 = L.spec.mode == "w8a8"
        if w8:
            codes, g = wq.wq_quantize_activations_w8a8(w, h["x"], stream)
            sf = xo = u = None
        else:
            codes, sf, g, xo, u = wq.wq_quantize_activations(h["w"], h["x"], wq.WQ_SCALE_LAYOUT_MMA, stream)
        torch.cuda.synchronize()

        def quant_fn(w=w, h=h, codes=codes, sf=sf, g=g, xo=xo, u=u, w8=w8):
            if w8:
                wq.lib().wq_quantize_activations_w8a8(ctypes.c_void_p(w.handle), ctypes.c_void_p(h["x"].data_ptr()),
                                                      M, ctypes.c_void_p(codes.data_ptr()),
                                                      ctypes.c_void_p(g.data_ptr()),
                                                      ctypes.c_void_p(stream.cuda_stream))
            else:
                wq.wq_quantize_activations_into(w, h["x"], codes, sf, g, xo, u, stream)

        def gemm_fn(w=w, h=h, codes=codes, sf=sf, g=g, xo=xo, u=u):
            wq.wq_linear_forward_quantized(w, codes, sf, g, u, xo, h["y"], stream)

        spec = L.spec
        for kname, fn in (("quant", quant_fn), ("gemm", gemm_fn)):
            fn()                                            # warm (tensor maps cached)
            times = queued_event_times(fn, iters, stream, flush)
            ms = statistics.median(times)
            if kname == "gemm":
                byts = gemm8_algorithmic_bytes(M, spec.K, spec.N, L.bias is not None) if w8 else \
                    gemm_algorithmic_bytes(M, spec.K, spec.N, L.rank, L.omega.size, L.bias is not None)
                flops = 2.0 * M * spec.K * spec.N
                kern = {wq.WQ_GEMM_WIDE: "wide_gemm_kernel", wq.WQ_GEMM_WIDE_DB: "wide_db_gemm_kernel"}.get(
                    wq.wq_gemm_schedule(w, M), "nvfp4_gemm_kernel")
            else:
                byts = quant8_algorithmic_bytes(M, spec.K, L.s is not None) if w8 else \
                    quant_algorithmic_bytes(M, spec.K, L.rank, L.omega.size, L.s is not None)
                flops = 0.0
                kern = {wq.WQ_QUANT_STREAM: "quantize_stream_kernel", wq.WQ_QUANT_RESIDENT: "quantize_resident_kernel"
                        }.get(wq.wq_quant_schedule(w, M), "quantize_kernel")
            rl = kernel_roofline(flops, byts, ms, peaks)
            per_kernel.append(dict(name=f"{kname}[{spec.name}]", kernel=kern, ms=ms, bytes=byts, flops=flops,
                                   spread_us=[1e3 * min(times), 1e3 * max(times)], **rl))
    dom = max(per_kernel, key=lambda k: k["ms"])
    tot_ms = sum(k["ms"] for k in per_kernel)
    if dom["bound"] == "tensor":
        ach = dom["flops"] / (dom["ms"] / 1e3) / 1e12
        peak, unit, src = fp4_peak_tflops(peaks), "TFLOP/s", \
            f"{peak_kind} bf16 burst {peaks.get('bf16_tflops')} TFLOP/s x 6 (nominal fp4 : bf16 ratio)"
    else:
        ach = dom["bytes"] / (dom["ms"] / 1e3) / 1e9
        peak, unit, src = peaks["hbm_gbs"], "GB/s", f"{peak_kind} HBM copy bandwidth"
    try:
        mb_tf, mb_ns, mb_mhz = wq.wq_mma_peak("fp4", 256, True, 0, 0, 8192, 0, False, 1)
        microbench = {"tflops": mb_tf, "ns_per_mma": mb_ns, "sm_mhz": mb_mhz,
                      "form": "tcgen05.mma.cta_group::2 kind::mxf4nvf4 M256 N256 K64, no scale copies"}
    except Exception as exc:  # reported, not hidden
        microbench = {"error": repr(exc)}
    if "tflops" in microbench:
        # each contraction's rate against the tensor pipe's measured FP4 issue rate as well
        gemms = [k for k in per_kernel if k["flops"]]
        microbench["frac_by_kernel"] = {k["name"]: k["flops"] / (k["ms"] / 1e3) / 1e12 / microbench["tflops"]
                                        for k in gemms}
    roofline = {"kernel": f"{dom['name']} {dom['kernel']}", "bound": dom["bound"], "achieved": ach, "peak": peak,
                "unit": unit, "frac": ach / peak,
                "traffic": profiled_traffic(dom["kernel"], args.workload),
                "peak_source": src,
                "bytes_per_launch": dom["bytes"], "flops_per_launch": dom["flops"],
                "us_per_launch": 1e3 * dom["ms"], "share_of_kernel_time": dom["ms"] / tot_ms,
                "step": {"roofline_us": sum(k["roofline_us"] for k in per_kernel), "measured_us": 1e3 * tot_ms,
                         "frac": sum(k["roofline_us"] for k in per_kernel) / (1e3 * tot_ms)},
                "fp4_mma_microbench": microbench}
    kernels = {k["name"]: {"kernel": k["kernel"], "us": 1e3 * k["ms"], "min_max_us": k["spread_us"],
                           "bytes": k["bytes"], "flops": k["flops"], "bound": k["bound"],
                           "roofline_us": k["roofline_us"], "frac": k["frac"],
                           "GB/s": k["bytes"] / (k["ms"] / 1e3) / 1e9,
                           "TFLOP/s": k["flops"] / (k["ms"] / 1e3) / 1e12} for k in per_kernel}

    # ---------------- end to end through the host-buffer entry point
    e2e = None
    try:
        hb = []
        for h in H:
            L = h["L"]
            xh = h["x"].cpu().pin_memory()
            yh = torch.empty((M, L.spec.N), dtype=torch.bfloat16).pin_memory()
            wsh = torch.empty(wq.wq_host_workspace_bytes(h["w"], M), dtype=torch.uint8, device=dev)
            hb.append((h["w"], xh, yh, wsh))
        ke = max(10, min(K, 500))
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ke)]
        with torch.cuda.stream(stream):
            for i in range(ke + 3):
                flush.zero_()
                if i >= 3:
                    evs[i - 3][0].record(stream)
                for w, xh, yh, wsh in hb:
                    wq.wq_linear_forward_host(w, xh, yh, wsh, stream)
                if i >= 3:
                    evs[i - 3][1].record(stream)
        torch.cuda.synchronize()
        e_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        e2e = {"value": M * ws / (e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(2 * M * h["L"].spec.K for h in H),
               "d2h_bytes_per_step": sum(2 * M * h["L"].spec.N for h in H),
               "ms_per_step": e_ms, "api": "wq_linear_forward_host (pinned host x and y)"}
    except Exception as exc:  # reported, not hidden
        e2e = {"value": None, "unit": "tokens/s", "error": repr(exc)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        n_threads = os.cpu_count() or 1
        try:
            tps, rows, passes, el = time_oracle(layers, args.cpu_baseline_seconds, n_threads,
                                                fp8=args.workload == "backbone_fp8")
            cpu = {"value": tps, "unit": "tokens/s", "cores": n_threads, "kind": "oracle",
                   "sample": f"{rows} of {M} rows x {passes} passes over all {len(layers)} layers "
                             f"({el:.1f} s, weights prepared beforehand)"}
        except Exception as exc:
            cpu = {"value": None, "error": repr(exc)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 (e2m1 x e2m1, ue4m3 scales, f32 accumulate)", "data": "synthetic (seeded)",
            "tflops": tflops,
            "config": {"workload": WORKLOAD_TEXT[args.workload], "M": M,
                       "layers": [f"{h['L'].spec.name} {h['L'].spec.K}->{h['L'].spec.N}" for h in H],
                       "l2": "flushed before every step (256 MiB write, outside the step events)",
                       "parallelism": f"replicas x{ws}", "cuda_graph": True},
            "roofline": roofline, "kernels": kernels,
            "cpu_baseline": cpu, "e2e": e2e,
            "clocks": sampler.record(),
            "gpu_launches": launches_per_step * K,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_conv(args):
    """The VAE Conv3d workload: one step = |x| maxima + voxel quantiser + implicit GEMM."""
    import torch
    ws_, rank, local_rank = dist_env()
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from w4a4_nvfp4_quantized_wq_b300 import build as wqbuild
    wqbuild.build_library()
    import w4a4_nvfp4_quantized_wq_b300 as wq
    import workloads as wl
    xb, w = wl.make_conv_inputs()
    _, C, D, H, W = xb.shape
    V, N, K = D * H * W, w.shape[0], 27 * C
    hw = wq.wq_prepare_conv3d(w)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.empty((1, N, D, H, W), dtype=torch.bfloat16, device=dev)
    wsb = torch.empty(wq.wq_conv3d_workspace_bytes(hw, 1, D, H, W), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        wq.wq_conv3d_forward(hw, x, y, wsb, stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            wq.wq_conv3d_forward(hw, x, y, wsb, stream)
    torch.cuda.synchronize()
    wq.wq_check_device_error(hw)
    Ksteps, Wu = args.steps, args.warmup
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ksteps)]
    with torch.cuda.stream(stream):
        for _ in range(Wu):
            flush.zero_()
            graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    if ws_ > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with sampler:
        with torch.cuda.stream(stream):
            for i in range(Ksteps):
                flush.zero_()
                ev[i][0].record(stream)
                graph.replay()
                ev[i][1].record(stream)
        torch.cuda.synchronize()
    total_ms = job_time_ms(float(sum(a.elapsed_time(b) for a, b in ev)), ws_, dev)
    flops = 2.0 * V * N * K
    # per-kernel: the quantiser pair alone, the whole forward; the GEMM is the difference
    import ctypes
    codes = torch.empty((V, C // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((V, C // 16), dtype=torch.uint8, device=dev)
    gx = torch.empty(1, dtype=torch.float32, device=dev)

    def quant_fn():
        wq.lib().wq_quantize_conv3d_input(
            ctypes.c_void_p(hw.handle), ctypes.c_void_p(x.data_ptr()), 1, D, H, W,
            ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
            ctypes.c_void_p(gx.data_ptr()), ctypes.c_void_p(wsb.data_ptr()), wsb.numel(),
            ctypes.c_void_p(stream.cuda_stream))

    def fwd_fn():
        wq.wq_conv3d_forward(hw, x, y, wsb, stream)

    times = {"quant": statistics.median(queued_event_times(quant_fn, args.kernel_iters, stream, flush)),
             "forward": statistics.median(queued_event_times(fwd_fn, args.kernel_iters, stream, flush))}
    gemm_ms = times["forward"] - times["quant"]
    peaks, peak_kind = measured_peaks()
    fp4_peak = fp4_peak_tflops(peaks)
    ach = flops / (gemm_ms / 1e3) / 1e12
    qbytes = 2 * 2 * C * V + V * C // 2 + V * C // 16          # x read twice (maxima + quantiser), codes out
    gbytes = V * C // 2 + V * C // 16 + N * K // 2 + N * K // 16 + 2 * N * V   # codes in (once), weights, y out
    rl = kernel_roofline(flops, gbytes, gemm_ms, peaks)
    roofline = {"kernel": "conv_gemm_kernel", "bound": rl["bound"], "achieved": ach, "peak": fp4_peak,
                "unit": "TFLOP/s", "frac": ach / fp4_peak, "traffic": profiled_traffic("conv_gemm_kernel", "vae_conv"),
                "peak_source": f"{peak_kind} bf16 burst {peaks.get('bf16_tflops')} TFLOP/s x 6 (nominal fp4 : bf16 ratio)",
                "flops_per_launch": flops, "bytes_per_launch": gbytes, "us_per_launch": 1e3 * gemm_ms,
                "share_of_kernel_time": gemm_ms / times["forward"]}
    kernels = {"conv_quant (maxima + quantiser)": {"us": 1e3 * times["quant"], "bytes": qbytes,
                                                    "GB/s": qbytes / (times["quant"] / 1e3) / 1e9},
               "conv_gemm (forward - quantiser)": {"us": 1e3 * gemm_ms, "TFLOP/s": ach, **rl}}
    # end to end: pinned host x -> device, forward, y -> pinned host
    xh = x.cpu().pin_memory()
    yh = torch.empty(y.shape, dtype=torch.bfloat16).pin_memory()
    ke = max(5, min(Ksteps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ke)]
    with torch.cuda.stream(stream):
        for i in range(ke):
            flush.zero_()
            evs[i][0].record(stream)
            x.copy_(xh, non_blocking=True)
            wq.wq_conv3d_forward(hw, x, y, wsb, stream)
            yh.copy_(y, non_blocking=True)
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    e_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and ws_ == 1:
        import oracle
        nth = os.cpu_count() or 1
        vox = np.sort(np.random.default_rng(5).choice(V, 16, replace=False))
        t0 = time.perf_counter()
        passes = 0
        while True:
            oracle.conv3d_reference(xb, w, vox, nth)
            passes += 1
            if time.perf_counter() - t0 > args.cpu_baseline_seconds * 0.5:
                break
        el = time.perf_counter() - t0
        cpu = {"value": 16 * passes / el, "unit": "voxels/s", "cores": nth, "kind": "oracle",
               "sample": f"16 of {V} output voxels x {passes} passes, all 384 channels, input and weight "
                         f"quantisation included ({el:.1f} s)"}
    if rank == 0:
        line = {"metric": METRIC, "value": job_throughput(V, Ksteps, ws_, total_ms), "unit": "voxels/s",
                "n_gpus": ws_, "steps": Ksteps, "warmup": Wu, "ms_per_step": total_ms / Ksteps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "nvfp4 (e2m1 x e2m1, ue4m3 scales, f32 accumulate)", "data": "synthetic (seeded)",
                "tflops": flops * Ksteps * ws_ / (total_ms / 1e3) / 1e12,
                "config": {"workload": WORKLOAD_TEXT["vae_conv"], "M": V, "N": N, "K": K,
                           "l2": "flushed before every step (256 MiB write, outside the step events)",
                           "parallelism": f"replicas x{ws_}", "cuda_graph": True},
                "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu,
                "e2e": {"value": V * ws_ / (e_ms / 1e3), "unit": "voxels/s",
                        "h2d_bytes_per_step": 2 * C * V, "d2h_bytes_per_step": 2 * N * V, "ms_per_step": e_ms,
                        "api": "pinned host x -> device, wq_conv3d_forward, y -> pinned host"},
                "clocks": sampler.record(), "gpu_launches": 3 * Ksteps}
        print(json.dumps(line), flush=True)


def run_mma_peak(args):
    """Tensor-core issue rate of each instruction form the kernels use (one JSON line)."""
    import torch
    torch.cuda.set_device(0)
    from w4a4_nvfp4_quantized_wq_b300 import build as wqbuild
    wqbuild.build_library()
    import w4a4_nvfp4_quantized_wq_b300 as wq
    rows = []
    # (kind, N, pair, copies per MMA, copy shape, feeder, zero operands, accumulators)
    forms = [("fp4", 256, True, 0, 0, 0, 0, 1), ("fp4", 256, False, 0, 0, 0, 0, 1), ("fp4", 128, False, 0, 0, 0, 0, 1),
             ("fp4", 128, True, 0, 0, 0, 0, 1), ("fp4", 192, False, 0, 0, 0, 0, 1), ("fp4", 64, False, 0, 0, 0, 0, 1),
             ("bf16", 256, False, 0, 0, 0, 0, 1), ("bf16", 128, False, 0, 0, 0, 0, 1), ("bf16", 256, True, 0, 0, 0, 0, 1),
             ("fp8", 256, False, 0, 0, 0, 0, 1), ("fp8", 256, True, 0, 0, 0, 0, 1),
             ("fp4", 256, False, 0, 0, 0, 1, 1), ("fp8", 256, False, 0, 0, 0, 1, 1), ("bf16", 256, False, 0, 0, 0, 1, 1),
             ("fp4", 128, False, 0, 0, 0, 0, 2), ("fp8", 256, False, 0, 0, 0, 0, 2), ("bf16", 256, False, 0, 0, 0, 0, 2),
             ("fp4", 256, True, 3, 0, 0, 0, 1), ("fp4", 256, False, 1, 0, 0, 0, 1), ("fp4", 256, False, 3, 0, 0, 0, 1),
             ("fp4", 256, False, 1, 1, 0, 0, 1), ("fp4", 256, True, 1, 1, 0, 0, 1),
             ("fp4", 256, False, 1, 0, 1, 0, 1), ("fp4", 256, False, 3, 0, 1, 0, 1), ("fp4", 256, True, 3, 0, 1, 0, 1),
             ("fp4", 256, False, 1, 0, 2, 0, 1), ("fp4", 256, False, 3, 0, 2, 0, 1)]
    for kind, n, pair, copies, shape, feeder, zero, accs in forms:
        best = None
        for _ in range(3):
            t, ns, mhz = wq.wq_mma_peak(kind, n, pair, copies, shape, 8192, feeder, zero, accs)
            if best is None or t > best[0]:
                best = (t, ns, mhz)
        rows.append({"kind": kind, "M": 256 if pair else 128, "N": n, "cta_pair": pair, "copies_per_mma": copies,
                     "copy_shape": ["32x128b.warpx4", "128x256b"][shape],
                     "feeder": ["mma thread", "other warp", "tcgen05.st warps"][feeder], "zero_operands": bool(zero),
                     "accumulators": accs, "tflops": best[0], "ns_per_mma": best[1], "sm_mhz": best[2]})
    peaks, kind_ = measured_peaks()
    print(json.dumps({"mma_peak": rows, "bf16_cublas_tflops": peaks.get("bf16_tflops"), "peaks": kind_}), flush=True)


def main():
    args = parse_args()
    if args.mma_peak:
        run_mma_peak(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.workload == "vae_conv":
        run_conv(args)
    else:
        run_wq(args)


if __name__ == "__main__":
    main()
