"""Measure the tensor core's dense FP8 and block-scaled FP8 / FP4 rates.

    python -m fp4_gemm_gb300.peak [--iters 65536] [--reps 20]

Runs the library's bsg_mma_peak microbenchmark (every SM issuing
back-to-back tcgen05.mma from shared memory, no global traffic) for each
kind, times each launch with CUDA events on the launching stream, samples
the SM clock with nvidia-smi meanwhile, and prints one JSON line:
{"kind/pair": {"tflops": median, "best_tflops": ..., "sm_mhz": median}, ...}.
"""
from __future__ import annotations

import argparse
import json
import statistics
import subprocess
import time

import torch

import fp4_gemm_gb300 as bsg

KINDS = [("e4m3", False, False), ("e4m3", False, True), ("e4m3", True, False),
         ("e2m1", True, False), ("e2m1", True, True)]


def measure(fmt, block_scaled, pair, iters, reps):
    stream = torch.cuda.current_stream()
    bsg.bsg_mma_peak(fmt, pair, 64, block_scaled=block_scaled)
    torch.cuda.synchronize()
    times, flops = [], 0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        flops = bsg.bsg_mma_peak(fmt, pair, iters, block_scaled=block_scaled)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3)
    if bsg.bsg_device_error() != 0:
        raise RuntimeError("bsg_mma_peak reported a device error")
    times.sort()
    return flops / times[len(times) // 2] / 1e12, flops / times[0] / 1e12


def peaks(iters=1 << 16, reps=20, clocks=True):
    out = {}
    for fmt, bs, pair in KINDS:
        proc = None
        if clocks:
            try:
                f = open("/tmp/bsg_peak_clocks.csv", "w")
                proc = subprocess.Popen(["nvidia-smi", "--query-gpu=clocks.sm", "--format=csv,noheader,nounits",
                                         "-lms", "20"], stdout=f, stderr=subprocess.DEVNULL)
                time.sleep(0.1)
            except OSError:
                proc = None
        med, best = measure(fmt, bs, pair, iters, reps)
        mhz = None
        if proc is not None:
            proc.terminate()
            proc.wait()
            f.close()
            vals = [float(x) for x in open("/tmp/bsg_peak_clocks.csv") if x.strip()]
            mhz = statistics.median(vals) if vals else None
        name = {("e4m3", False): "fp8_dense", ("e4m3", True): "mxfp8", ("e2m1", True): "mxfp4"}[(fmt, bs)]
        out[f"{name}{'/pair' if pair else ''}"] = {"tflops": round(med, 1), "best_tflops": round(best, 1),
                                                   "sm_mhz": mhz}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--iters", type=int, default=1 << 16)
    ap.add_argument("--reps", type=int, default=20)
    a = ap.parse_args()
    bsg.load_library()
    print(json.dumps(peaks(a.iters, a.reps)))


if __name__ == "__main__":
    main()
