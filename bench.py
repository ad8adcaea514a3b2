"""Benchmark of the block-scaled GEMM hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Workloads (synthetic, seeded; see synth/):
  ffn_up      FP8 FFN-up GEMM, M=8192 tokens, K=4096, N=14336.  One step =
              quantise the FP32 activations to E4M3 with 1x128 scales, then the
              promoted FP8 GEMM against pre-quantised E4M3 weights (128x128
              scales), BF16 output.  Metric TFLOP/s (2MNK per step).   [default]
  dgrad       FP8 dgrad GEMM, M=8192, K=14336, N=4096: E5M2 gradients (128x128
              scales, quantised in the step) x E4M3 weights, FP32 output.
  decode      MXFP4 decode, M=16 (or --m 1), K=8192, N=28672: quantise the BF16
              activations to MXFP4, then the decode-shaped GEMM against
              pre-quantised MXFP4 weights, BF16 out.  Metric GB/s of algorithmic
              bytes (weights + scales + activations + output).
  fp8_256, mxfp4_1024   the small parity configurations (latency-bound).
  mxfp8_ffn_up  the FFN-up shape and inputs with MXFP8 operands (E4M3, one
              E8M0 scale per 32 along K, applied by the tensor core, so the
              GEMM needs no promotion): quantise the activations with the MX
              rule, then the block-scaled FP8 GEMM, BF16 out.
  nvfp4_ffn_up  the FFN-up shape with NVFP4 operands (E2M1, one E4M3 scale per
              16 along K, FP32 tensor scales: 1 for the activations, 2^-6
              for the weights): quantise the activations, then the block-
              scaled FP4 GEMM (alpha = 2^-6), BF16 out.
  bs16_ffn_up  the FFN-up shape with E2M1 operands and one BF16 scale per
              32 along K ("Rubin FP4 GEMM deep dive" section 3.2): quantise
              the activations, then the GEMM that promotes every 32-wide K
              block's partial on CUDA cores, BF16 out.  Its roofline is the
              FP32 pipe (two FP32 operations per output per K block).
  ffn_up_q8out  the FFN-up step with the quantiser fused into the GEMM's
              epilogue: the output leaves as E4M3 codes with one FP32 scale
              per 1x128 run of a row (the next GEMM's activation operand)
              instead of BF16.  Same FLOPs; output bytes 1 + 4/128 per element.

One JSON line is printed by rank 0.  Timing: W warm-up steps, then K steps.
For the three full-size workloads every input and output exists in several
copies (together more than twice the 129 MB L2) and consecutive steps use
consecutive copies, so no step finds its data in L2; the K steps run back to
back as replays of a CUDA graph of one step per copy, and one pair of CUDA
events on the launching stream brackets all of them.  The small parity
configurations fit in L2 many times over, so each of their steps is one graph
replay bracketed by events with an L2 flush before it (a 256 MB write, then a
256 MB read), outside the events.  The GEMM alone is timed the same way for K
more steps (roofline).  `e2e` repeats the step through the same API
with the activations copied from pinned host memory and the output copied back
inside the timed region.  `cpu_baseline` times the CPU oracle on a bounded
sample of the same workload.  Under torchrun every rank runs an independent
replica ("replicas only": the path has no exchange step), value = sum over
ranks, time = max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense ratios to BF16 (2.25 PF): FP8 4.5 PF, FP4 13.5 PF
RATIO = {"fp8": 2.0, "fp4": 6.0}
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {"fp8": ["gemm_fp8.cu", "common.cuh", "quant_math.cuh"], "fp4": ["gemm_mxfp4.cu", "common.cuh", "quant_math.cuh"],
                  "mx": ["gemm_mx.cu", "common.cuh"], "bs16": ["gemm_bs16.cu", "common.cuh"]}
# workloads that reuse another workload's shape and seeded inputs
SHAPE_OF = {"mxfp8_ffn_up": "ffn_up", "ffn_up_q8out": "ffn_up", "nvfp4_ffn_up": "ffn_up",
            "bs16_ffn_up": "ffn_up"}


def kernel_source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "fp4_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, kind):
    """DRAM bytes per launch of the workload's GEMM from the committed ncu
    summary, or None when there is none or the kernel source changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            entry = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not entry or entry.get("src_sha") != kernel_source_hash(KERNEL_SOURCES[kind]):
        return None
    return entry.get("dram_bytes")


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="ffn_up",
                    choices=["ffn_up", "dgrad", "decode", "fp8_256", "mxfp4_1024", "mxfp8_ffn_up",
                             "ffn_up_q8out", "nvfp4_ffn_up", "bs16_ffn_up"])
    ap.add_argument("--m", type=int, default=None, help="override M (e.g. 1 for decode)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------- workload
class Workload:
    """Inputs and one step of the hot path for a named workload."""

    def __init__(self, name, m_override, dev):
        import torch
        import fp4_gemm_gb300 as bsg
        self.bsg, self.torch, self.dev, self.name = bsg, torch, dev, name
        src = SHAPE_OF.get(name, name)
        idx, M, N, K = synth.WORKLOADS[src]
        if m_override is not None:
            M = m_override
        self.M, self.N, self.K = M, N, K
        A, B = synth.make(src, m=M)
        self.fp4 = name in ("decode", "mxfp4_1024")
        self.mx8 = name == "mxfp8_ffn_up"
        self.q8out = name == "ffn_up_q8out"
        self.nv4 = name == "nvfp4_ffn_up"
        self.bs16 = name == "bs16_ffn_up"
        # decode: the BF16 activations are quantised on the fly inside one
        # API call (bsg_gemm_mxfp4_act); up to four rows in the GEMM kernel
        # itself, above that by the quantiser launched first
        self.act = name == "decode"
        self.act_fused = self.act and M <= 4
        self.launches_per_step = 1 if self.act_fused else 2
        self.g_a, self.g_b = 1.0, 2.0 ** -6      # NVFP4 tensor scales
        if name == "ffn_up":
            self.fa, self.fb, self.ga, self.gb, self.out = "e4m3", "e4m3", "row", "tile", "bf16"
        elif self.q8out:
            self.fa, self.fb, self.ga, self.gb, self.out = "e4m3", "e4m3", "row", "tile", "e4m3/row"
        elif self.nv4:
            self.fa, self.fb, self.ga, self.gb, self.out = "e2m1", "e2m1", "nv", "nv", "bf16"
        elif self.bs16:
            self.fa, self.fb, self.ga, self.gb, self.out = "e2m1", "e2m1", "bf16", "bf16", "bf16"
        elif name == "dgrad":
            self.fa, self.fb, self.ga, self.gb, self.out = "e5m2", "e4m3", "tile", "tile", "f32"
        elif name == "fp8_256":
            self.fa, self.fb, self.ga, self.gb, self.out = "e4m3", "e4m3", "tile", "tile", "f32"
        elif name == "mxfp4_1024":
            self.fa, self.fb, self.ga, self.gb, self.out = "e2m1", "e2m1", "mx", "mx", "f32"
        elif name == "mxfp8_ffn_up":
            self.fa, self.fb, self.ga, self.gb, self.out = "e4m3", "e4m3", "mx", "mx", "bf16"
        else:
            self.fa, self.fb, self.ga, self.gb, self.out = "e2m1", "e2m1", "mx", "mx", "bf16"
        self.A_host = A
        if name == "decode":
            bits = synth.to_bf16_bits(A)
            self.A_host_t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        else:
            self.A_host_t = torch.from_numpy(A).pin_memory()
        A0 = self.A_host_t.to(dev)
        Bt = torch.from_numpy(B).to(dev)
        # weights are quantised once, outside the step (static parameters)
        if self.nv4:
            qb, sb = bsg.bsg_quantize_nvfp4(Bt, "tcgen05", tensor_scale=self.g_b)
        elif self.bs16:
            qb, sb = bsg.bsg_quantize_fp4_bs16(Bt, "bf16")
        elif self.fp4:
            qb, sb = bsg.bsg_quantize_mxfp4(Bt, "tcgen05")
        elif self.mx8:
            qb, sb = bsg.bsg_quantize_mx(Bt, self.fb, "tcgen05")
        else:
            qb, sb = bsg.bsg_quantize_fp8(Bt, self.fb, self.gb)
        del Bt
        # Timed steps cycle over `sets` copies of every input and output, so
        # no step finds its data in L2 (the copies together exceed twice the
        # 129 MB L2); tiny workloads use one set and an explicit L2 flush.
        touched = self.step_bytes()
        self.rotating = touched >= (8 << 20)
        self.nsets = max(2, -(-2 * L2_BYTES // int(touched)) + 1) if self.rotating else 1
        self.sets = []
        for r in range(self.nsets):
            st = {"A": A0 if r == 0 else A0.clone(),
                  "qb": qb if r == 0 else qb.clone(), "sb": sb if r == 0 else sb.clone()}
            if self.nv4:
                st["qa"], st["sa"] = bsg.bsg_quantize_nvfp4(st["A"], "tcgen05", tensor_scale=self.g_a)
            elif self.bs16:
                st["qa"], st["sa"] = bsg.bsg_quantize_fp4_bs16(st["A"], "bf16")
            elif self.fp4:
                st["qa"], st["sa"] = bsg.bsg_quantize_mxfp4(st["A"], "tcgen05")
            elif self.mx8:
                st["qa"], st["sa"] = bsg.bsg_quantize_mx(st["A"], self.fa, "tcgen05")
            else:
                st["qa"], st["sa"] = bsg.bsg_quantize_fp8(st["A"], self.fa, self.ga)
            if self.q8out:
                st["D"] = torch.empty((M, N), dtype=torch.uint8, device=dev)
                st["sD"] = torch.empty(((N + 127) // 128, M), dtype=torch.float32, device=dev)
            else:
                st["D"] = torch.empty((M, N), dtype=torch.bfloat16 if self.out == "bf16" else torch.float32,
                                      device=dev)
            self.sets.append(st)
        self.A, self.D = self.sets[0]["A"], self.sets[0]["D"]
        self.D_host = torch.empty_like(self.D, device="cpu").pin_memory()
        self.sD_host = torch.empty_like(self.sets[0]["sD"], device="cpu").pin_memory() if self.q8out else None
        self.ws = bsg.workspace_for(M, N, K, self.fa, self.fb, dev)
        if self.act:
            n = max(bsg.bsg_gemm_mxfp4_act_workspace_size(M, N, K), 16)
            self.ws_act = torch.zeros((n,), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def quantize(self, r=0):
        b, st = self.bsg, self.sets[r]
        if self.nv4:
            b.bsg_quantize_nvfp4(st["A"], "tcgen05", tensor_scale=self.g_a, q=st["qa"], sf=st["sa"])
        elif self.bs16:
            b.bsg_quantize_fp4_bs16(st["A"], "bf16", q=st["qa"], sf=st["sa"])
        elif self.fp4:
            b.bsg_quantize_mxfp4(st["A"], "tcgen05", q=st["qa"], sf=st["sa"])
        elif self.mx8:
            b.bsg_quantize_mx(st["A"], self.fa, "tcgen05", q=st["qa"], sf=st["sa"])
        else:
            b.bsg_quantize_fp8(st["A"], self.fa, self.ga, q=st["qa"], scales=st["sa"])

    def act_gemm(self, r=0):
        st = self.sets[r]
        self.bsg.bsg_gemm_mxfp4_act(st["A"], st["qb"], st["sb"], out=self.out, D=st["D"],
                                    workspace=self.ws_act)

    def gemm(self, r=0):
        st = self.sets[r]
        if self.act_fused:        # the dominant kernel is the fused call itself
            self.act_gemm(r)
            return
        if self.nv4:
            self.bsg.bsg_gemm_nvfp4(st["qa"], st["sa"], st["qb"], st["sb"], alpha=self.g_a * self.g_b,
                                    out=self.out, D=st["D"], K=self.K)
            return
        if self.q8out:
            self.bsg.bsg_gemm_quantized(st["qa"], self.fa, st["sa"], self.ga, st["qb"], self.fb, st["sb"],
                                        self.gb, qfmt="e4m3", Dq=st["D"], sD=st["sD"])
            return
        self.bsg.bsg_gemm(st["qa"], self.fa, st["sa"], self.ga, st["qb"], self.fb, st["sb"], self.gb,
                          out=self.out, D=st["D"], workspace=self.ws, K=self.K)

    def step(self, r=0):
        if self.act:
            self.act_gemm(r)
            return
        self.quantize(r)
        self.gemm(r)

    # algorithmic quantities
    def flops(self):
        return 2.0 * self.M * self.N * self.K

    def gemm_bytes(self):
        """Bytes a GEMM must move at least once: operands, scales, output."""
        M, N, K = self.M, self.N, self.K
        if self.nv4:
            a = M * K / 2 + M * K / 16
            b = N * K / 2 + N * K / 16
        elif self.bs16:
            a = M * K / 2 + M * K / 32 * 2
            b = N * K / 2 + N * K / 32 * 2
        elif self.fp4:
            # fused decode: the kernel reads the BF16 activations themselves
            a = M * K * 2 if self.act_fused else M * K / 2 + M * K / 32
            b = N * K / 2 + N * K / 32
        elif self.mx8:
            a = M * K + M * K / 32
            b = N * K + N * K / 32
        else:
            a = M * K + (M * -(-K // 128) * 4 if self.ga == "row" else 4 * -(-M // 128) * -(-K // 128))
            b = N * K + 4 * -(-N // 128) * -(-K // 128)
        if self.q8out:
            d = M * N + 4 * M * -(-N // 128)
        else:
            d = M * N * (2 if self.out == "bf16" else 4)
        return a + b + d

    def step_bytes(self):
        """Algorithmic bytes of a whole step (quantiser read + write, GEMM)."""
        if self.act_fused:
            return self.gemm_bytes()          # the activations are read once, by the GEMM
        src = self.M * self.K * (2 if self.name == "decode" else 4)
        return src + self.gemm_bytes()

    def metric(self):
        if self.name == "decode":
            return "GB/s of algorithmic bytes (decode M<=16, % of HBM)", "GB/s"
        return "GEMM TFLOP/s (% of GB300 dense FP8/FP4 peak)", "TFLOP/s"

    def value_from_seconds(self, sec):
        if self.name == "decode":
            return self.step_bytes() / sec / 1e9
        return self.flops() / sec / 1e12


# ------------------------------------------------------------- clock sampler
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"bsg_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    smax = float(c[2])
                    power.append(float(c[3]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons)}
        loaded = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- CPU baseline
def host_cores():
    """Host CPUs this process may run on (its affinity mask, which honours
    cgroup and taskset limits), not the machine's total."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count()


def cpu_baseline(name, m_override, target_s=15.0):
    """The CPU oracle as it stands, on a bounded sample of the workload."""
    import oracle.gemm as og
    import oracle.quantize as oq
    idx, M, N, K = synth.WORKLOADS[SHAPE_OF.get(name, name)]
    if m_override is not None:
        M = m_override
    cores = host_cores()
    if name == "decode":
        # a slice of the weight rows: quantise + GEMM, scaled to the metric (GB/s)
        nrows = 4096
        A, B = synth.make(name, m=M, n=nrows, k=K)
        A = synth.bf16_bits_to_f32(synth.to_bf16_bits(A))
        t0 = time.perf_counter()
        pa, fa = oq.quantize_mxfp4(A)
        pb, fb = oq.quantize_mxfp4(B)
        og.gemm_mxfp4(pa, fa, pb, fb)
        dt = time.perf_counter() - t0
        nbytes = nrows * K / 2 + nrows * K / 32 + M * K * 2 + M * nrows * 2
        return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
                "sample": f"decode M={M}, {nrows} of {N} weight rows, K={K}: oracle quantise + GEMM, "
                          f"{dt:.1f} s"}
    if name == "mxfp8_ffn_up":
        # the MX oracle picks every block's scale in a Python loop: a slice of
        # B's rows keeps the sample bounded
        rows, ncols = 128, 2048
        A, B = synth.make("ffn_up", m=rows, n=ncols)
        t0 = time.perf_counter()
        qa, sfa = oq.quantize_mxfp8(A, "e4m3")
        qb, sfb = oq.quantize_mxfp8(B, "e4m3")
        og.gemm_mxfp8(qa, "e4m3", sfa, qb, "e4m3", sfb)
        dt = time.perf_counter() - t0
        return {"value": 2.0 * rows * ncols * K / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{name}: {rows} of {M} rows of A with {ncols} of {N} rows of B (K={K}); "
                          f"oracle MXFP8 quantise (both operands) + FP64 GEMM, {dt:.1f} s"}
    if name == "nvfp4_ffn_up":
        rows, ncols = 128, 2048
        A, B = synth.make("ffn_up", m=rows, n=ncols)
        t0 = time.perf_counter()
        pa, fa = oq.quantize_nvfp4(A)
        pb, fb = oq.quantize_nvfp4(B, tensor_scale=2.0 ** -6)
        og.gemm_nvfp4(pa, fa, pb, fb, alpha=2.0 ** -6)
        dt = time.perf_counter() - t0
        return {"value": 2.0 * rows * ncols * K / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{name}: {rows} of {M} rows of A with {ncols} of {N} rows of B (K={K}); "
                          f"oracle NVFP4 quantise (both operands) + FP64 GEMM, {dt:.1f} s"}
    if name == "bs16_ffn_up":
        rows, ncols = 128, 2048
        A, B = synth.make("ffn_up", m=rows, n=ncols)
        t0 = time.perf_counter()
        pa, fa = oq.quantize_fp4_bs16(A, "bf16")
        pb, fb = oq.quantize_fp4_bs16(B, "bf16")
        og.gemm_fp4_bs16(pa, fa, pb, fb, "bf16")
        dt = time.perf_counter() - t0
        return {"value": 2.0 * rows * ncols * K / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{name}: {rows} of {M} rows of A with {ncols} of {N} rows of B (K={K}); "
                          f"oracle FP4 + BF16-block-scale quantise (both operands) + FP64 GEMM, {dt:.1f} s"}
    if name == "ffn_up_q8out":
        rows = 128
        A, B = synth.make("ffn_up", m=rows)
        t0 = time.perf_counter()
        qa, sa = oq.quantize_fp8(A, "e4m3", "row")
        qb, sb = oq.quantize_fp8(B, "e4m3", "tile")
        D, _ = og.gemm_fp8(qa, "e4m3", sa, "row", qb, "e4m3", sb, "tile")
        oq.quantize_fp8(D.astype(np.float32), "e4m3", "row")
        dt = time.perf_counter() - t0
        return {"value": 2.0 * rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
                "kind": "oracle",
                "sample": f"{name}: {rows} of {M} rows of A with all of B (N={N}, K={K}); oracle "
                          f"quantise (both operands) + FP64 GEMM + 1x128 quantiser of the output, "
                          f"{dt:.1f} s"}
    fa, fb, ga, gb = {"ffn_up": ("e4m3", "e4m3", "row", "tile"),
                      "dgrad": ("e5m2", "e4m3", "tile", "tile"),
                      "fp8_256": ("e4m3", "e4m3", "tile", "tile"),
                      "mxfp4_1024": ("e2m1", "e2m1", "mx", "mx")}[name]
    rows = min(M, 128)
    A, B = synth.make(name, m=rows)
    t0 = time.perf_counter()
    if fa == "e2m1":
        pa, sfa = oq.quantize_mxfp4(A)
        pb, sfb = oq.quantize_mxfp4(B)
        og.gemm_mxfp4(pa, sfa, pb, sfb)
    else:
        qa, sa = oq.quantize_fp8(A, fa, ga)
        qb, sb = oq.quantize_fp8(B, fb, gb)
        og.gemm_fp8(qa, fa, sa, ga, qb, fb, sb, gb)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{name}: {rows} of {M} rows of A with all of B (N={N}, K={K}); oracle "
                      f"quantise (both operands) + FP64 GEMM, {dt:.1f} s"}


# -------------------------------------------------------------------- runs
def max_over_ranks(value, dist, device):
    """The largest of every rank's value (the job's time is its slowest
    rank's); `value` itself on a single process."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def run_reference(args, world, rank):
    if rank != 0:
        return
    cb = cpu_baseline(args.workload, args.m, target_s=10.0)
    vals = []
    for _ in range(args.warmup):
        pass
    for _ in range(max(1, min(args.steps, 3))):
        vals.append(cpu_baseline(args.workload, args.m)["value"])
    v = statistics.median(vals)
    idx, M, N, K = synth.WORKLOADS[SHAPE_OF.get(args.workload, args.workload)]
    metric = ("GB/s of algorithmic bytes (decode M<=16, % of HBM)" if args.workload == "decode"
              else "GEMM TFLOP/s (% of GB300 dense FP8/FP4 peak)")
    line = {"impl": "reference", "metric": metric, "value": v, "unit": cb["unit"],
            "n_gpus": world, "steps": len(vals), "warmup": args.warmup,
            "higher_is_better": True, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "M": args.m or M, "N": N, "K": K},
            "cpu_baseline": dict(cb, value=v),
            "e2e": {"value": v, "unit": cb["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local, dist = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        if dist is not None:
            dist.barrier()
        return

    import torch
    import fp4_gemm_gb300 as bsg
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    bsg.load_library()
    w = Workload(args.workload, args.m, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        # write a buffer larger than L2, then read another one, so the timed
        # step starts with none of its data in L2 and no dirty lines to evict
        flush.fill_(float(i))
        clean.sum()

    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 0)):
        w.step()
    torch.cuda.synchronize()
    if bsg.bsg_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    # The step (quantise + GEMM) and the GEMM alone are captured once as CUDA
    # graphs and replayed, so the device time excludes host launch gaps.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        return g

    K = args.steps
    R = w.nsets
    if w.rotating:
        # one graph runs R consecutive steps, each on its own input set
        g_step = capture(lambda: [w.step(r) for r in range(R)])
        g_gemm = capture(lambda: [w.gemm(r) for r in range(R)])
        reps = -(-K // R)
    else:
        g_step = capture(w.step)
        g_gemm = capture(w.gemm)
        reps = K
    K = reps * R if w.rotating else K
    for _ in range(2):
        g_step.replay()
        g_gemm.replay()
    torch.cuda.synchronize()

    clocks = Clocks(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall0 = time.perf_counter()
    if w.rotating:
        # back-to-back replays; the whole timed region is one event pair
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        for _ in range(reps):
            g_step.replay()
        ev[1].record(stream)
        torch.cuda.synchronize()
        ev[2].record(stream)
        for _ in range(reps):
            g_gemm.replay()
        ev[3].record(stream)
        torch.cuda.synchronize()
        step_total = ev[0].elapsed_time(ev[1])
        gemm_total = ev[2].elapsed_time(ev[3])
        step_ms_mean = step_total / K
        gemm_ms_mean = gemm_total / K
        gemm_ms_min = gemm_ms_mean
    else:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        for i in range(K):
            flush_l2(i)                                 # outside the events
            ev[i][0].record(stream)
            g_step.replay()
            ev[i][1].record(stream)
        for i in range(K):
            flush_l2(i)
            ev[i][2].record(stream)
            g_gemm.replay()
            ev[i][3].record(stream)
        torch.cuda.synchronize()
        step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
        gemm_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
        step_ms_mean = statistics.mean(step_ms)
        gemm_ms_mean = statistics.mean(gemm_ms)
        gemm_ms_min = min(gemm_ms)
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    if bsg.bsg_device_error() != 0:
        raise RuntimeError("device error during the timed steps")
    ms = step_ms_mean
    ms = max_over_ranks(ms, dist, dev)

    # end to end through the API with host buffers (rotating over the same
    # input sets as the device-timed steps)
    e2e = None
    if not args.no_e2e:
        h2d = w.A_host_t.numel() * w.A_host_t.element_size()
        d2h = w.D.numel() * w.D.element_size()
        if w.q8out:
            d2h += w.sD_host.numel() * w.sD_host.element_size()

        # Three streams: the host->device copy of step i+1 and the
        # device->host copy of step i-1 run beside step i's kernels.  Step i
        # uses input/output set i % R (R >= 2): its input copy waits until
        # step i-R has finished reading that set, and its kernels wait until
        # the output of step i-R has left for the host.  Every copy of the K
        # steps lies inside the timed region.
        s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        D_hosts = [w.D_host] + [torch.empty_like(w.D_host).pin_memory() for _ in range(R - 1)]
        sD_hosts = ([w.sD_host] + [torch.empty_like(w.sD_host).pin_memory() for _ in range(R - 1)]
                    if w.q8out else None)

        def e2e_run(n, start_ev):
            for st_ in (s_h2d, s_cmp, s_d2h):
                st_.wait_event(start_ev)
            h2d_done, cmp_done, d2h_done = {}, {}, {}
            for i in range(n):
                r = i % R
                st = w.sets[r]
                with torch.cuda.stream(s_h2d):
                    if i >= R:
                        s_h2d.wait_event(cmp_done[i - R])
                    st["A"].copy_(w.A_host_t, non_blocking=True)
                    h2d_done[i] = torch.cuda.Event()
                    h2d_done[i].record(s_h2d)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(h2d_done[i])
                    if i >= R:
                        s_cmp.wait_event(d2h_done[i - R])
                    w.step(r)
                    cmp_done[i] = torch.cuda.Event()
                    cmp_done[i].record(s_cmp)
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(cmp_done[i])
                    D_hosts[r].copy_(st["D"], non_blocking=True)
                    if w.q8out:
                        sD_hosts[r].copy_(st["sD"], non_blocking=True)
                    d2h_done[i] = torch.cuda.Event()
                    d2h_done[i].record(s_d2h)
            for st_ in (s_h2d, s_cmp, s_d2h):
                stream.wait_stream(st_)

        warm = torch.cuda.Event()
        warm.record(stream)
        e2e_run(2 * R, warm)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(K, e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1) / K
        e_ms = max_over_ranks(e_ms, dist, dev)
        e2e = {"value": world * w.value_from_seconds(e_ms / 1e3), "unit": w.metric()[1],
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e_ms}

    pk, pk_kind = peaks()
    g_s = gemm_ms_mean / 1e3
    mp = None
    if w.name != "decode":
        # the tensor core's own rate for this kind, measured now on this GPU
        # (outside the timed region).  NVFP4 is timed against the MXFP4
        # microbenchmark: the peak tool has no scale_vec::4X kind.
        from fp4_gemm_gb300 import peak as mma_peak
        kind = ("e2m1", True) if (w.fp4 or w.nv4) else (("e4m3", True) if w.mx8 else ("e4m3", False))
        mp, _ = mma_peak.measure(kind[0], kind[1], False, 1 << 14, 5)
    if w.bs16:
        # The per-block promotion runs on the FP32 pipe: one multiply (s_A s_B)
        # and one FMA per output element per 32-wide K block; the tensor core
        # does 64 FLOPs in the same time and idles.  Peak = FP32 lanes x clock.
        ops = 2.0 * w.M * w.N * (w.K // 32)
        achieved = ops / g_s / 1e9
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clk.get("sm_mhz") or pk.get("sm_max_mhz", 2070.0)
        peak = sms * 128 * mhz / 1e3
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "G FP32 ops/s",
                "frac": achieved / peak, "traffic": measured_traffic(w.name, "bs16"),
                "kernel": "gemm_bs16_kernel",
                "peak_source": f"{sms} SMs x 128 FP32 lanes x {mhz:.0f} MHz (median SM clock "
                               "sampled during the timed region)",
                "tensor_tflops": w.flops() / g_s / 1e12, "mma_peak_microbench": mp}
    elif w.name == "decode":
        achieved = w.gemm_bytes() / g_s / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": measured_traffic(w.name, "fp4"),
                "kernel": "gemm_mxfp4_decode_kernel",
                "peak_source": f"{pk_kind} HBM copy bandwidth"}
    else:
        dt = "fp4" if (w.fp4 or w.nv4) else "fp8"
        achieved = w.flops() / g_s / 1e12
        derived = pk["bf16_tflops"] * RATIO[dt]
        # The denominator is the larger of the two ceilings: the measured
        # cuBLAS BF16 rate times the nominal dense ratio, and the tensor
        # core's own measured rate for this MMA kind.  The other one is kept
        # beside it.
        peak = max(derived, mp)
        derived_src = (f"{pk_kind} cuBLAS BF16 burst x {RATIO[dt]:g} (nominal dense "
                       f"{dt.upper()}:BF16 ratio)")
        mp_src = "tcgen05 MMA-rate microbenchmark of this kind on this GPU, measured after the timed region"
        # MXFP8 and the large NVFP4 GEMM run the 128 x 256 block-scaled kernel
        src_kind = "mx" if (w.mx8 or w.nv4) else dt
        kernel = "gemm_mxfp4_kernel" if w.fp4 else ("gemm_mx_kernel" if (w.mx8 or w.nv4) else "gemm_fp8_kernel")
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": measured_traffic(w.name, src_kind),
                "kernel": kernel,
                "peak_source": mp_src if mp >= derived else derived_src,
                "peak_cublas_derived": derived, "frac_of_cublas_derived": achieved / derived,
                "mma_peak_microbench": mp, "frac_of_mma_peak_microbench": achieved / mp}
    metric, unit = w.metric()
    value = world * w.value_from_seconds(ms / 1e3)
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1" if (w.fp4 or w.nv4 or w.bs16) else (w.fa if w.fa == w.fb else f"{w.fa}x{w.fb}"),
        "data": "synthetic (seeded; weights random-init and pre-quantised)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K,
                   "a": f"{w.fa}/{w.ga}", "b": f"{w.fb}/{w.gb}", "out": w.out,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"inputs rotate over {R} copies ({R} x {w.step_bytes() / 1e6:.0f} MB > L2): "
                          "no step finds its data in L2" if w.rotating else
                          "flushed before every timed step (256 MB write, then a 256 MB read)"),
                   "timing": ("one CUDA-event pair around K back-to-back steps (CUDA graphs of "
                              f"{R} steps replayed)" if w.rotating else
                              "CUDA events around a CUDA-graph replay of each step")},
        "quantize_ms": max(step_ms_mean - gemm_ms_mean, 0.0), "gemm_ms": gemm_ms_mean,
        "gemm_ms_min": gemm_ms_min,
        "wall_s": wall,
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": (w.launches_per_step + 1) * K,   # K steps + K GEMM-only launches
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.m)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
