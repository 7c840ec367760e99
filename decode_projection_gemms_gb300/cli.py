"""Run and time one skinny GEMM shape, or the KDA projection, with the
library's choice of kernel.

    python -m decode_projection_gemms_gb300.cli --M 4096 --N 4096 --K 7168 [--reps 5]
        [--cfg kind=cc,split_k=2,block=256,rows=4,k_unroll=1]
    python -m decode_projection_gemms_gb300.cli --kda --M 1 16 128 [--layers 4] [--reps 1]

GEMM: prints the configuration used (the table's or the built-in rule's
choice, or the one given with --cfg as comma-separated kp_cfg fields) and the
device time per call over `reps` calls after one warm-up call, with CUDA
events on the launching stream. --kda: the projection of the pages' shapes
(packed [4096 + 136, 7168] weight, W_fb [1024, 128]) for each M in the
table's mode, eagerly, `reps` passes over a stack of `layers` weight layers
(one layer per call; 4 layers are 244 MB, above the L2). Inputs are seeded
synthetic bf16 (or fp16 with --fp16).
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


def run_kda(m_list, layers: int, reps: int):
    from .inputs import gen_kda_layer
    dev = torch.device("cuda", torch.cuda.current_device())
    K, Nq, Nfab, Nfb = 7168, 4096, 136, 1024
    stack = [tuple(t.to(dev) for t in gen_kda_layer(layer, seed=0, device="cpu" if layer == 0 else dev))
             for layer in range(layers)]
    plan = binding.KdaPlan(K, Nq, Nfab, Nfb, max_M=max(m_list))
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    stream = torch.cuda.current_stream()
    try:
        for M in m_list:
            x = gen_x(M, K, seed=0, device=dev)
            outs = plan.outputs(M, dev)
            plan.run(x, *stack[0], *outs, aux_stream=aux, events=evs)   # warm-up
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                for wp, wfb in stack:
                    plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
            b.record(stream)
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / (reps * layers)
            print(json.dumps({"M": M, "mode": plan.overlap_at(M), "us_per_call_eager": round(us, 3),
                              "configs": {br: plan.get_config(i, M).as_dict()
                                          for i, br in enumerate(("qkvg", "fab", "fb"))},
                              "device_error": binding.device_error()}))
    finally:
        plan.close()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--kda", action="store_true", help="run the KDA projection instead of one GEMM")
    ap.add_argument("--M", type=int, nargs="+", required=True)
    ap.add_argument("--N", type=int)
    ap.add_argument("--K", type=int)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--fp16", action="store_true")
    ap.add_argument("--residual", action="store_true")
    ap.add_argument("--cfg", default=None, help="explicit configuration, e.g. kind=cc,split_k=2")
    args = ap.parse_args(argv)
    cfg_in = parse_cfg(args.cfg) if args.cfg else None

    build()
    binding.load()
    if args.kda:
        run_kda(args.M, args.layers, args.reps)
        return
    if args.N is None or args.K is None or len(args.M) != 1:
        ap.error("a GEMM needs one --M and --N, --K")
    args.M = args.M[0]
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
