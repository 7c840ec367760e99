"""Run and time one skinny GEMM shape with the library's choice of kernel.

    python -m decode_projection_gemms_gb300.cli --M 4096 --N 4096 --K 7168 [--reps 5]

Prints the configuration the table (or the built-in rule) picks and the device
time per call over `reps` calls after one warm-up call, with CUDA events on the
launching stream. Inputs are seeded synthetic bf16 (or fp16 with --fp16).
"""
from __future__ import annotations

import argparse
import json

import torch

from . import binding
from .build import build
from .inputs import gen_w, gen_x


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--M", type=int, required=True)
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--K", type=int, required=True)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--fp16", action="store_true")
    ap.add_argument("--residual", action="store_true")
    args = ap.parse_args(argv)

    build()
    binding.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    dt = torch.float16 if args.fp16 else torch.bfloat16
    x = gen_x(args.M, args.K, seed=1, device=dev, dtype=dt)
    W = gen_w(args.N, args.K, seed=2, device=dev, dtype=dt)
    r = gen_x(args.M, args.N, seed=3, device=dev, dtype=dt) if args.residual else None
    y = torch.empty((args.M, args.N), dtype=dt, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cfg = binding.select_config(args.M, args.N, args.K, sms)
    stream = torch.cuda.current_stream()
    binding.skinny_gemm_ex(x, W, r, y)            # warm-up (attributes, scratch)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.reps):
        binding.skinny_gemm_ex(x, W, r, y)
    b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / args.reps
    flops = 2.0 * args.M * args.N * args.K
    nbytes = 2 * (args.M * args.K + args.N * args.K + args.M * args.N)
    print(json.dumps({"M": args.M, "N": args.N, "K": args.K, "config": cfg.as_dict(),
                      "us_per_call": round(us, 3), "tflops": round(flops / us / 1e6, 1),
                      "gbs": round(nbytes / us / 1e3, 1),
                      "device_error": binding.device_error()}))


if __name__ == "__main__":
    main()
