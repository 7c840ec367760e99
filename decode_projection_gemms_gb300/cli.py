"""Run and time one skinny GEMM shape with the library's choice of kernel.

    python -m decode_projection_gemms_gb300.cli --M 4096 --N 4096 --K 7168 [--reps 5]
        [--cfg kind=cc,split_k=2,block=256,rows=4,k_unroll=1]

Prints the configuration used (the table's or the built-in rule's choice, or
the one given with --cfg as comma-separated kp_cfg fields) and the device time
per call over `reps` calls after one warm-up call, with CUDA events on the
launching stream. Inputs are seeded synthetic bf16 (or fp16 with --fp16).
"""
from __future__ import annotations

import argparse
import json

import torch

from . import binding
from .binding import KpCfg
from .build import build
from .inputs import gen_w, gen_x

CFG_FIELDS = ("kind", "split_k", "block", "rows", "k_unroll", "producers", "stages", "flags")


def parse_cfg(text: str) -> KpCfg:
    """'kind=tc05,split_k=8,k_unroll=2' -> KpCfg (fields not given keep
    KpCfg.make's defaults)."""
    kw = {}
    for item in text.split(","):
        key, _, val = item.partition("=")
        key = key.strip()
        if key not in CFG_FIELDS or not val:
            raise ValueError(f"bad --cfg item {item!r}; fields: {', '.join(CFG_FIELDS)}")
        kw[key] = val.strip() if key == "kind" else int(val)
    if "kind" not in kw:
        raise ValueError("--cfg needs kind=cc|tc05|smallk")
    return KpCfg.make(**kw)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--M", type=int, required=True)
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--K", type=int, required=True)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--fp16", action="store_true")
    ap.add_argument("--residual", action="store_true")
    ap.add_argument("--cfg", default=None, help="explicit configuration, e.g. kind=cc,split_k=2")
    args = ap.parse_args(argv)
    cfg_in = parse_cfg(args.cfg) if args.cfg else None

    build()
    binding.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    dt = torch.float16 if args.fp16 else torch.bfloat16
    x = gen_x(args.M, args.K, seed=1, device=dev, dtype=dt)
    W = gen_w(args.N, args.K, seed=2, device=dev, dtype=dt)
    r = gen_x(args.M, args.N, seed=3, device=dev, dtype=dt) if args.residual else None
    y = torch.empty((args.M, args.N), dtype=dt, device=dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cfg = cfg_in if cfg_in is not None else binding.select_config(args.M, args.N, args.K, sms)
    stream = torch.cuda.current_stream()
    binding.skinny_gemm_ex(x, W, r, y, cfg=cfg_in)   # warm-up (attributes, scratch)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.reps):
        binding.skinny_gemm_ex(x, W, r, y, cfg=cfg_in)
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
