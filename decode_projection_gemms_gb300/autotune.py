"""Offline autotune sweep: measure candidate kernel configurations per
(M, N, K) and write the table the library loads (tune/gb300_table.txt).

Timing method: every candidate runs as a captured CUDA graph of `layers`
back-to-back calls, each on a different layer of a weight stack at least
4x the L2 size (cold weight reads from HBM, as in decode), replayed
`reps` times between CUDA events on the capturing stream; the result is the
median over `trials` of (elapsed / calls).

The table format is one line per measured (M, N, K):
    M N K kind split_k block rows k_unroll producers stages flags overlap
Usage (on a GB300):
    python -m decode_projection_gemms_gb300.autotune --shapes kda --out tune/gb300_table.txt
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import os
import statistics
import sys
import time

import torch

from . import binding
from .binding import KpCfg

L2_BYTES = 129 * 1024 * 1024

KDA_SHAPES = [(4096, 7168), (136, 7168), (1024, 128)]
SWEEP_M = list(range(1, 17)) + [24, 32, 48, 64, 96, 128, 129, 256]
SWEEP_N = [136, 512, 1024, 4096, 8192]
SWEEP_K = [128, 1024, 7168, 16384]


def cc_candidates(M: int, N: int, K: int, sms: int):
    out = []
    for (R, U) in ((1, 4), (2, 2), (2, 4), (4, 1), (4, 2), (8, 1)):
        for block in (128, 256):
            rows_cta = (block // 32) * R
            tiles = math.ceil(N / rows_cta)
            for waves in (1, 2, 4, 8):
                S = max(1, min(K // 256 if K >= 256 else 1, round(waves * sms / tiles)))
                out.append(KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U))
    # dedupe
    seen, uniq = set(), []
    for c in out:
        key = (c.split_k, c.block, c.rows, c.k_unroll)
        if key not in seen:
            seen.add(key)
            uniq.append(c)
    return uniq


def tc05_candidates(M: int, N: int, K: int, sms: int):
    out = []
    T = math.ceil(N / 128)
    for C in (1, 2, 4, 8, 16):
        if T * C > 2 * sms:
            continue
        for nkb in (1, 2, 4):
            for P in sorted({1, min(nkb, 2), nkb}):
                for stages in (0, 2, 3, 4):
                    out.append(KpCfg.make("tc05", split_k=C, k_unroll=nkb, producers=P,
                                          stages=stages))
    return out


def smallk_candidates(M: int, N: int, K: int, sms: int):
    return [KpCfg.make("smallk", block=b, rows=r) for b in (128, 256) for r in (8, 16, 32)]


def candidates(M, N, K, sms, kinds=("cc", "tc05", "smallk")):
    out = []
    if "smallk" in kinds and K <= 256:
        out += smallk_candidates(M, N, K, sms)
    if "cc" in kinds and M <= 16:
        out += cc_candidates(M, N, K, sms)
    if "tc05" in kinds:
        out += tc05_candidates(M, N, K, sms)
    valid = []
    for c in out:
        try:
            binding.scratch_bytes(M, N, K, c, sms)
            valid.append(c)
        except binding.KdaProjError:
            pass
    return valid


class Bench:
    """Weight stack + graph timing for one (M, N, K)."""

    def __init__(self, M, N, K, device, min_layers=4, seed=0):
        self.M, self.N, self.K = M, N, K
        per = N * K * 2
        self.layers = max(min_layers, math.ceil(4 * L2_BYTES / per))
        self.layers = min(self.layers, 256)
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.W = (torch.randn((self.layers, N, K), generator=g, device=device) * 0.02).to(torch.bfloat16)
        self.x = torch.randn((M, K), generator=g, device=device).to(torch.bfloat16)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.stream = torch.cuda.Stream(device=device)

    def time_cfg(self, cfg, reps=10, trials=3):
        with torch.cuda.stream(self.stream):
            binding.skinny_gemm(self.x, self.W[0], self.y, cfg=cfg)  # warm (scratch, attributes)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for l in range(self.layers):
                binding.skinny_gemm(self.x, self.W[l], self.y, cfg=cfg)
        res = []
        with torch.cuda.stream(self.stream):
            g.replay()
            for _ in range(trials):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(self.stream)
                for _ in range(reps):
                    g.replay()
                b.record(self.stream)
                b.synchronize()
                res.append(a.elapsed_time(b) * 1e3 / (reps * self.layers))
        del g
        return statistics.median(res)

    def bytes(self):
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


def sweep_shape(M, N, K, sms, device, kinds, verbose=False):
    b = Bench(M, N, K, device)
    results = []
    for c in candidates(M, N, K, sms, kinds):
        try:
            us = b.time_cfg(c)
        except binding.KdaProjError as e:
            if verbose:
                print(f"  skip {c.as_dict()}: {e}", file=sys.stderr)
            continue
        results.append((us, c))
        if verbose:
            print(f"  M={M} N={N} K={K} {us:8.3f} us {b.bytes() / us / 1e3:7.1f} GB/s {c.as_dict()}",
                  file=sys.stderr)
    results.sort(key=lambda r: r[0])
    del b
    torch.cuda.empty_cache()
    return results


def table_line(M, N, K, cfg, overlap=1, us=None):
    kind = binding.KIND_NAMES[cfg.kind]
    s = (f"{M} {N} {K} {kind} {cfg.split_k} {cfg.block} {cfg.rows} {cfg.k_unroll} {cfg.producers} "
         f"{cfg.stages} {cfg.flags} {overlap}")
    return s + (f"  # {us:.3f} us" if us is not None else "")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default="kda", help="kda | sweep | N:K[,N:K...]")
    ap.add_argument("--m", type=int, nargs="*", default=None)
    ap.add_argument("--kinds", default="cc,tc05,smallk")
    ap.add_argument("--out", default=None)
    ap.add_argument("--json", default=None)
    ap.add_argument("--top", type=int, default=3)
    ap.add_argument("-v", action="store_true")
    args = ap.parse_args(argv)

    from .build import build
    build()
    binding.load()
    binding.table_clear()
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if args.shapes == "kda":
        shapes = KDA_SHAPES
        ms = args.m or [1, 2, 4, 8, 16, 32, 64, 128]
    elif args.shapes == "sweep":
        shapes = [(n, k) for n in SWEEP_N for k in SWEEP_K]
        ms = args.m or SWEEP_M
    else:
        shapes = [tuple(int(v) for v in s.split(":")) for s in args.shapes.split(",")]
        ms = args.m or [1, 2, 4, 8, 16, 32, 64, 128]
    kinds = tuple(args.kinds.split(","))
    lines, dump = [], []
    t0 = time.time()
    for (N, K) in shapes:
        for M in ms:
            res = sweep_shape(M, N, K, sms, dev, kinds, args.v)
            if not res:
                continue
            best_us, best = res[0]
            lines.append(table_line(M, N, K, best, 1, best_us))
            dump.append({"M": M, "N": N, "K": K,
                         "results": [{"us": us, **c.as_dict()} for us, c in res[:args.top]]})
            print(lines[-1], flush=True)
    print(f"# sweep took {time.time() - t0:.1f} s", file=sys.stderr)
    if args.out:
        with open(args.out, "w") as f:
            f.write("# kdaproj autotune table v1 (measured on "
                    f"{torch.cuda.get_device_name(dev)}, {sms} SMs)\n")
            f.write("# Each line: M N K kind split_k block rows k_unroll producers stages flags overlap\n")
            f.write("# A call with (M, N, K) takes the entry with the same (N, K) and the smallest\n")
            f.write("# M >= its own; shapes without an entry use the library's built-in rule.\n")
            for l in lines:
                f.write(l + "\n")
    if args.json:
        with open(args.json, "w") as f:
            json.dump(dump, f, indent=1)


if __name__ == "__main__":
    main()
