#!/usr/bin/env python3
"""Benchmark of the tiled GEMM library on GB300.

Default workload: one square GEMM M = N = K = 4096, FP16 operands drawn from
U[-1, 1) (seeded), FP32 accumulation, FP16 output -- 137.4 GFLOP per call.
A "step" is one call of the library's C ABI (``tg_gemm``) on that problem.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Measurement:
  * inputs are resident in HBM before the timed region; each step uses the
    next of R rotating (A, B, C) sets whose total exceeds twice the L2 size, so
    no step finds its operands in L2;
  * the timed region is K back-to-back steps with torch.cuda.synchronize() on
    both sides, timed with CUDA events recorded on the stream the kernels are
    launched on;
  * ``roofline.achieved`` divides the algorithmic FLOPs of one launch (2MNK) by
    the average duration of a launch in the timed region (its length over K;
    no events between launches, which would block the overlap of consecutive
    launches);
  * ``e2e`` repeats the workload through ``tg_gemm_host`` with pinned HOST
    buffers: the host->device copies of A and B and the device->host copy of C
    (pipelined with the multiply by the library) are inside its timed region;
  * SM clocks and throttle reasons are sampled with nvidia-smi during the timed
    region;
  * ``cpu_baseline`` times the CPU FP64 oracle on a
    bounded sample of output rows of the same problem.

``--impl reference`` runs the CPU oracle arm instead (rank 0 only under
torchrun); each step is a bounded sample of output rows of the same workload.

One GPU only.  The library's tile kernels share A tiles between the CTAs of
a cluster by TMA multicast, which is only used in single-GPU processes: the
GPU arm refuses ``--gpus`` > 1 and a torchrun launch with WORLD_SIZE > 1.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (FP16/BF16 at 4096³) and % of GB300 dense tensor peak, 1 GPU"

WORKLOADS = {
    # name: (M, N, K, dtype_in, dtype_out, dist, description)
    "small127_f16": (127, 255, 65, "f16", "f32", "uniform",
                     "ragged 127x255x65, FP16 in U[-1,1), FP32 out (the correctness case)"),
    "square256_f16": (256, 256, 256, "f16", "f16", "uniform",
                      "square GEMM 256^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "square512_f16": (512, 512, 512, "f16", "f16", "uniform",
                      "square GEMM 512^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "square1024_f16": (1024, 1024, 1024, "f16", "f16", "uniform",
                       "square GEMM 1024^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "square2048_f16": (2048, 2048, 2048, "f16", "f16", "uniform",
                       "square GEMM 2048^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "square4096_f16": (4096, 4096, 4096, "f16", "f16", "uniform",
                       "square GEMM 4096^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "panel1024x4096x4096_f16": (1024, 4096, 4096, "f16", "f16", "uniform",
                                "row panel 1024x4096x4096 FP16 (the product tg_gemm_host runs "
                                "per panel of a 4096^3 call)"),
    "square8192_f16": (8192, 8192, 8192, "f16", "f16", "uniform",
                       "square GEMM 8192^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "square16384_f16": (16384, 16384, 16384, "f16", "f16", "uniform",
                        "square GEMM 16384^3, FP16 in U[-1,1), FP32 accumulate, FP16 out"),
    "prefill_qkv_bf16": (8192, 6144, 4096, "bf16", "bf16", "normal",
                         "prefill QKV projection 8192x6144x4096, BF16 in N(0,0.02), BF16 out"),
    "prefill_o_bf16": (8192, 4096, 4096, "bf16", "bf16", "normal",
                       "prefill output projection 8192x4096x4096, BF16 N(0,0.02)"),
    "prefill_up_bf16": (8192, 14336, 4096, "bf16", "bf16", "normal",
                        "prefill MLP up/gate (each) 8192x14336x4096, BF16 N(0,0.02)"),
    "prefill_down_bf16": (8192, 4096, 14336, "bf16", "bf16", "normal",
                          "prefill MLP down 8192x4096x14336, BF16 N(0,0.02)"),
    "square4096_e4m3": (4096, 4096, 4096, "e4m3", "f16", "uniform",
                        "square GEMM 4096^3, FP8 E4M3 in U[-1,1), FP32 accumulate, FP16 out"),
    "square8192_e4m3": (8192, 8192, 8192, "e4m3", "f16", "uniform",
                        "square GEMM 8192^3, FP8 E4M3 in U[-1,1), FP32 accumulate, FP16 out"),
    "tf32_2048": (2048, 2048, 2048, "f32", "f32", "uniform",
                  "FP32 operands at TF32 2048^3, FP32 out"),
    "tf32_ragged": (1000, 1999, 777, "f32", "f32", "uniform",
                    "FP32 operands at TF32, ragged 1000x1999x777 (tails in M, N and K), "
                    "FP32 out"),
    "skinny1_f16": (1, 8192, 8192, "f16", "f16", "uniform", "skinny M=1, N=K=8192 FP16"),
    "skinny16_f16": (16, 8192, 8192, "f16", "f16", "uniform", "skinny M=16, N=K=8192 FP16"),
    "skinny64_f16": (64, 8192, 8192, "f16", "f16", "uniform", "skinny M=64, N=K=8192 FP16"),
    "skinny128_f16": (128, 8192, 8192, "f16", "f16", "uniform", "skinny M=128, N=K=8192 FP16"),
    "skinny1_e4m3": (1, 8192, 8192, "e4m3", "f16", "uniform",
                     "skinny M=1, N=K=8192, FP8 E4M3 operands, FP16 out"),
    "skinny128_e4m3": (128, 8192, 8192, "e4m3", "f16", "uniform",
                       "skinny M=128, N=K=8192, FP8 E4M3 operands, FP16 out"),
    # strided batches (one tg_gemm_strided_batched call; contiguous [batch, rows, cols])
    "batched16x2048_f16": (2048, 2048, 2048, "f16", "f16", "uniform",
                           "strided batch of 16 GEMMs 2048^3, FP16 in U[-1,1), FP16 out"),
    "batched64x1024_bf16": (1024, 1024, 1024, "bf16", "bf16", "normal",
                            "strided batch of 64 GEMMs 1024^3, BF16 N(0,0.02)"),
    "batched32x64x8192_f16": (64, 8192, 8192, "f16", "f16", "uniform",
                              "strided batch of 32 small-M GEMMs 64x8192x8192, FP16"),
    # the fused epilogue and the 3xTF32 mode
    "square4096_f16_bias_silu": (4096, 4096, 4096, "f16", "f16", "uniform",
                                 "square GEMM 4096^3 FP16 with a fused epilogue: "
                                 "silu(C + bias[n]), bias FP32 U[-1,1)"),
    "square4096_f32_3xtf32": (4096, 4096, 4096, "f32", "f32", "uniform",
                              "square GEMM 4096^3, FP32 operands as three TF32 products "
                              "(near-FP32 accuracy), FP32 out"),
}
# planner options and fused epilogues that are part of a workload's definition
WORKLOAD_OPTS = {"square4096_f32_3xtf32": {"f32_mode": 1}}
WORKLOAD_EPILOGUE = {"square4096_f16_bias_silu": {"activation": "silu", "bias": True}}
# tensor FLOPs the method performs per algorithmic 2MNK (3xTF32: three TF32 products)
TENSOR_WORK = {"square4096_f32_3xtf32": 3.0}
# products per call of the batched workloads (1 for every other workload)
BATCH = {"batched16x2048_f16": 16, "batched64x1024_bf16": 64, "batched32x64x8192_f16": 32}
DEFAULT_WORKLOAD = "square4096_f16"
ESIZE = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}
# dense tensor-core peak of an operand type relative to BF16 (nominal ratios of
# 4.5 : 2.25 : 1.1 PFLOP/s for FP8 : BF16 : TF32)
PEAK_RATIO = {"f16": 1.0, "bf16": 1.0, "f32": 0.5, "e4m3": 2.0, "e5m2": 2.0}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------- plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


ONE_GPU_ONLY = ("the GPU arm runs on one GPU only: its tile kernels share A tiles inside a "
                "cluster by TMA multicast, which this library uses only in single-GPU "
                "processes (got {what})")


def refuse_multi_gpu(gpus: int, world: int):
    """The reason the GPU arm refuses this launch, or None for one GPU."""
    if gpus > 1:
        return ONE_GPU_ONLY.format(what=f"--gpus {gpus}")
    if world > 1:
        return ONE_GPU_ONLY.format(what=f"WORLD_SIZE={world}")
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Sources that define the kernels (the tile kernel and the small-M kernel with
# the headers they share); a DRAM-traffic figure is valid only for the hash
# it was captured on.
KERNEL_SOURCES = ("gemm_tc_kernel.cuh", "gemm_skinny_kernel.cuh", "tg_epilogue.cuh",
                  "tg_kernel_common.cuh", "tg_ptx.cuh", "tg_internal.h")


def _code_only(text: str) -> str:
    """C/C++ source without comments and blank lines (string and character
    literals kept as they are), so that edits to comments leave the hash of
    the kernel code unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(ch)
            i += 1
    lines = (ln.rstrip() for ln in "".join(out).splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tiled_matrix_multiplication_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(workload)
    if not ent or ent.get("source_sha") != kernel_source_sha():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def _gpu_id(self):
        try:
            import torch
            p = torch.cuda.get_device_properties(self.dev)
            return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:  # noqa: BLE001
            return str(self.dev)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self._gpu_id()],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ oracle (CPU)

def oracle_rate(M, N, K, din, dist, rows: int, seed_rows=12345):
    """Time the FP64 oracle on `rows` sampled output rows; returns
    (TFLOP/s, seconds, threads)."""
    import numpy as np

    import oracle
    from tiled_matrix_multiplication_gb300 import inputs
    rng = np.random.default_rng(seed_rows)
    sel = np.sort(rng.choice(M, size=min(rows, M), replace=False))
    a_rows = np.concatenate([inputs.matrix_bits(1, K, din, dist, inputs.SEED_A, row_start=int(r))
                             for r in sel])
    b = inputs.matrix_bits(K, N, din, dist, inputs.SEED_B)
    oracle.build()
    t0 = time.perf_counter()
    oracle.gemm_ref_bits(a_rows, b, K=K, N=N, fmt=din)
    dt = time.perf_counter() - t0
    return 2.0 * len(sel) * N * K / dt / 1e12, dt, oracle.num_threads()


def cpu_baseline(M, N, K, din, dist, target_s=10.0):
    rate, dt, thr = oracle_rate(M, N, K, din, dist, rows=8)
    per_row = dt / 8
    rows = int(max(8, min(M, target_s / max(per_row, 1e-9))))
    rate, dt, thr = oracle_rate(M, N, K, din, dist, rows=rows)
    return {"value": rate, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": f"{rows} seeded output rows x all {N} columns of the {M}x{N}x{K} problem "
                      f"({dt:.1f} s, FP64 three-loop oracle incl. decoding B)"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    M, N, K, din, dout, dist, desc = WORKLOADS[args.workload]
    _, dt0, thr = oracle_rate(M, N, K, din, dist, rows=4)
    per_row = dt0 / 4
    budget = 120.0
    rows = int(max(1, min(M, budget / max(per_row * (args.steps + args.warmup), 1e-9))))
    for _ in range(args.warmup):
        oracle_rate(M, N, K, din, dist, rows=rows)
    times = []
    for s in range(args.steps):
        _, dt, thr = oracle_rate(M, N, K, din, dist, rows=rows, seed_rows=1000 + s)
        times.append(dt)
    total = sum(times)
    value = 2.0 * rows * N * K * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "M": M, "N": N, "K": K, "batch": BATCH.get(args.workload, 1),
                   "dtype_in": din, "dtype_out": dout,
                   "step": f"{rows} sampled output rows of the problem"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                         "sample": f"{rows} seeded output rows x {N} columns per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm

def run_ours(args, local):
    import numpy as np
    import torch

    import tiled_matrix_multiplication_gb300 as tg
    from tiled_matrix_multiplication_gb300 import build as tgbuild
    from tiled_matrix_multiplication_gb300 import inputs

    torch.cuda.set_device(local)
    tgbuild.build()
    tg.load()
    M, N, K, din, dout, dist, desc = WORKLOADS[args.workload]
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
           "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
    iview = {"f16": np.int16, "bf16": np.int16, "f32": np.int32, "e4m3": np.uint8,
             "e5m2": np.uint8}

    nb = BATCH.get(args.workload, 1)
    a_bits = np.stack([inputs.matrix_bits(M, K, din, dist, inputs.SEED_A + z) for z in range(nb)])
    b_bits = np.stack([inputs.matrix_bits(K, N, din, dist, inputs.SEED_B + z) for z in range(nb)])
    a_host = torch.from_numpy(a_bits.view(iview[din])).view(tdt[din])
    b_host = torch.from_numpy(b_bits.view(iview[din])).view(tdt[din])
    set_bytes = nb * ((M * K + K * N) * ESIZE[din] + M * N * ESIZE[dout])
    R = max(2, -(-2 * l2 // set_bytes) + 1)
    A0 = a_host.cuda()
    B0 = b_host.cuda()
    sets = []
    for i in range(R):
        sets.append((A0 if i == 0 else A0.clone(), B0 if i == 0 else B0.clone(),
                     torch.empty((nb, M, N), dtype=tdt[dout], device="cuda")))
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    code_in, code_out = tg.dtype_code(din), tg.dtype_code(dout)

    opts = dict(WORKLOAD_OPTS.get(args.workload, {}))
    opts.update({k: int(v) for k, v in (kv.split("=") for kv in args.opt)})
    topt = tg.make_options(**opts) if opts else None
    epi = None
    epi_spec = WORKLOAD_EPILOGUE.get(args.workload)
    if epi_spec is not None:
        bias_bits = inputs.matrix_bits(1, N, "f32", "uniform", 72)
        bias_d = torch.from_numpy(bias_bits.view(np.float32)[0].copy()).cuda()
        epi = tg.make_epilogue(bias=bias_d.data_ptr() if epi_spec.get("bias") else 0,
                               activation=epi_spec["activation"])
    if nb > 1:
        plan = tg.plan_batched(nb, M, N, K, din, dout, num_sms=props.multi_processor_count,
                               **opts)
    else:
        plan = tg.plan(M, N, K, din, dout, num_sms=props.multi_processor_count, **opts)

    def call(a, b, c):
        if epi is not None:
            return tg.tg_gemm_fused(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                                    code_in, code_out, epi, sh, topt)
        if nb > 1:
            return tg.tg_gemm_strided_batched(nb, M, N, K, a.data_ptr(), K, M * K, b.data_ptr(),
                                              N, K * N, c.data_ptr(), N, M * N, code_in,
                                              code_out, sh, topt)
        if topt is None:
            return tg.tg_gemm(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                              code_in, code_out, sh)
        return tg.tg_gemm_ex(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
                             code_in, code_out, sh, topt)

    def step(i):
        a, b, c = sets[i % R]
        st = call(a, b, c)
        if st != tg.TG_OK:
            raise tg.TgError(st, "tg_gemm")

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    tg.check_device_error()

    K_steps = args.steps
    # One event pair around the K back-to-back steps on the launching stream:
    # events between launches would stop a launch from starting its prologue
    # while the previous one drains (programmatic dependent launch), which for
    # a 15-25 us small-M launch costs a quarter of its time.  The average
    # launch duration is the region over K.
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)                                   # let nvidia-smi start sampling
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    ev_start.record(stream)
    for i in range(K_steps):
        step(i)
    ev_end.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    tg.check_device_error()
    region_ms = ev_start.elapsed_time(ev_end)
    kernel_ms = region_ms / K_steps

    flops = 2.0 * M * N * K * nb
    ms_per_step = region_ms / K_steps
    value = flops / (ms_per_step * 1e-3) / 1e12

    # ---- end to end through the C ABI with pinned host buffers
    e2e_steps = max(3, min(K_steps, 50))
    a_pin = a_host.pin_memory()
    b_pin = b_host.pin_memory()
    # two host result buffers and two streams, used alternately: step i+1's
    # host->device copies may then run while step i's result is still being
    # copied back (the library orders each call on its own stream only)
    c_pins = [torch.empty((nb, M, N), dtype=tdt[dout]).pin_memory() for _ in range(2)]
    e2e_streams = [stream, torch.cuda.Stream()]
    a_e, b_e, c_e = sets[0]

    def e2e_step(i):
        c_pin = c_pins[i % 2]
        st_handle = e2e_streams[i % 2].cuda_stream
        if epi is not None:
            # (tg_gemm_host has no epilogue: copy in, fused multiply, copy back)
            a_e.copy_(a_pin, non_blocking=True)
            b_e.copy_(b_pin, non_blocking=True)
            st = call(a_e, b_e, c_e)
            if st != tg.TG_OK:
                raise tg.TgError(st, "tg_gemm_fused")
            c_pin.copy_(c_e, non_blocking=True)
            return
        # tg_gemm_host: host operands in, host result out, copies pipelined
        # with the multiply inside the library
        st = tg.TG_OK
        for z in range(nb):
            st = tg.tg_gemm_host(M, N, K, a_pin.data_ptr() + z * M * K * ESIZE[din], K,
                                 b_pin.data_ptr() + z * K * N * ESIZE[din], N,
                                 c_pin.data_ptr() + z * M * N * ESIZE[dout], N, code_in,
                                 code_out, st_handle, topt)
            if st != tg.TG_OK:
                break
        if st != tg.TG_OK:
            raise tg.TgError(st, "tg_gemm_host")

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_streams[1].wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(e2e_streams[1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    tg.check_device_error()
    h2d = nb * (M * K + K * N) * ESIZE[din]
    d2h = nb * M * N * ESIZE[dout]

    pk, pk_kind = peaks()
    skinny = M <= 128
    if skinny:
        bound, unit = "hbm", "GB/s"
        alg = nb * ((M * K + K * N) * ESIZE[din] + M * N * ESIZE[dout])
        achieved = alg / (kernel_ms * 1e-3) / 1e9
        peak = float(pk["hbm_gbs"])
    else:
        bound, unit = "tensor", "TFLOP/s"
        achieved = TENSOR_WORK.get(args.workload, 1.0) * flops / (kernel_ms * 1e-3) / 1e12
        peak = float(pk["bf16_tflops"]) * PEAK_RATIO[din]
    roof = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": profiled_traffic(args.workload),
            "peak_source": f"{pk_kind} ({'hbm_gbs' if skinny else 'bf16_tflops'} burst"
                           f"{'' if skinny or PEAK_RATIO[din] == 1.0 else f', x{PEAK_RATIO[din]} nominal ratio to BF16'})",
            "tensor_flops_per_useful_flop": TENSOR_WORK.get(args.workload, 1.0),
            "kernel": ("gemm_skinny_kernel" if plan["path"] == tg.TG_PATH_SKINNY else "gemm_tc_kernel")
                      + ("" if plan["kernels"] == 1 else " (+ helper kernels)"),
            "launch_ms": round(kernel_ms, 5)}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": K_steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": din,
        "data": "synthetic",
        "config": {"workload": desc, "M": M, "N": N, "K": K, "batch": nb, "dtype_in": din,
                   "dtype_out": dout, "accumulate": "f32", "parallelism": "single",
                   "l2": f"{R} rotating input sets of {set_bytes / 1e6:.1f} MB "
                         f"(> 2x L2 {l2 / 1e6:.0f} MB)",
                   "tile": f"{plan['block_m']}x{plan['block_n']}x{plan['block_k']}",
                   "splits": plan["splits"], "ctas": plan["ctas"],
                   "multicast": plan["multicast"], "options": opts or None},
        "pct_of_peak": round(100.0 * value / peak, 2) if not skinny else None,
        "clocks": clocks,
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "how": ("tg_gemm_fused after host->device copies, result copied back"
                        if epi is not None else
                        "tg_gemm_host on pinned host buffers, steps alternating between two "
                        "streams")},
        "gpu_launches": K_steps * plan["kernels"],
        "roofline": roof,
        "wall_s": round(t_wall, 3),
        "gpu": props.name,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(M, N, K, din, dist, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--opt", action="append", default=[], metavar="KEY=VALUE",
                    help="planner override passed to tg_gemm_ex (tg_options field), e.g. "
                         "multicast=1; repeatable")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    why = refuse_multi_gpu(args.gpus, world)
    if why is not None:
        log("bench.py: " + why)
        return 2
    return run_ours(args, local)


if __name__ == "__main__":
    sys.exit(main())
