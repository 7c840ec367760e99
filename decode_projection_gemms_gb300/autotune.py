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
        for block in (128, 256, 512):
            rows_cta = (block // 32) * R
            tiles = math.ceil(N / rows_cta)
            for waves in (1, 2, 4, 8):
                S = max(1, min(K // 256 if K >= 256 else 1, round(waves * sms / tiles)))
                out.append(KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U))
    # Tiles sized for whole waves: for one or two CTAs per SM and S K slices,
    # the rows per CTA (whole warps of R rows) that bring tiles x S closest to
    # SMs x CTAs-per-SM without a partial wave.
    for (R, U) in ((1, 4), (2, 4), (2, 2), (4, 1), (4, 2)):
        for occ in (1, 2):
            for S in (1, 2, 3, 4):
                if S > max(1, K // 256):
                    continue
                target = max(1, sms * occ // S)
                warps = math.ceil(math.ceil(N / target) / R)
                block = 32 * warps
                if 32 <= block <= 512 // occ:
                    out.append(KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U))
    # each also in the shared-memory ring form (stages = 4), where it fits
    out += [KpCfg.make("cc", split_k=c.split_k, block=c.block, rows=c.rows, k_unroll=c.k_unroll, stages=4)
            for c in list(out)]
    # dedupe
    seen, uniq = set(), []
    for c in out:
        key = (c.split_k, c.block, c.rows, c.k_unroll, c.stages)
        if key not in seen:
            seen.add(key)
            uniq.append(c)
    return uniq


def tc05_candidates(M: int, N: int, K: int, sms: int):
    out = []
    for rows in (128, 256):   # feature rows per CTA (256: two accumulators share x)
        T = math.ceil(N / rows)
        for C in (1, 2, 4, 8, 16):
            if T * C > 2 * sms:
                continue
            for nkb in (1, 2, 4):
                # more producer warps where one CTA per SM streams W and x
                ps = {1, min(nkb, 2), nkb} | ({3, 5} if M >= 32 and nkb >= 2 else set())
                for P in sorted(ps):
                    for stages in (0, 2, 3, 4):
                        out.append(KpCfg.make("tc05", split_k=C, rows=rows, k_unroll=nkb,
                                              producers=P, stages=stages))
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
        _refuse_if_gave_up(cfg)
        return statistics.median(res)

    def bytes(self):
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


def sweep_candidates(M: int, N: int, K: int, sms: int):
    """A short list for the shape sweep: the settings that decided the
    projection shapes' tuning (grids of one to two CTAs per SM, split-K to fill
    them, two K blocks per stage, as many stages as fit), 10 to 30 per shape
    (the CUDA-core kernel's ring form adds up to 17 at M <= 16)."""
    out = []
    if K <= 256:
        out += [KpCfg.make("smallk", block=256, rows=r) for r in (8, 16)]
    if M <= 16:
        for (R, U, block) in ((1, 4, 256), (2, 4, 256), (4, 2, 256), (1, 4, 512), (2, 4, 512)):
            if R * M > 64:
                continue
            tiles = math.ceil(N / (block // 32 * R))
            for waves in (1, 2, 4):
                S = max(1, min(max(1, K // 256), round(waves * sms / tiles)))
                out.append(KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U))
        # the shared-memory ring form: 128- and 256-thread CTAs and CTAs sized
        # so that two per SM make whole waves
        for (R, U) in ((1, 4), (2, 2), (4, 1)) if M > 4 else ((1, 4), (2, 2)):
            for S in (1, 2):
                if S > max(1, K // 256):
                    continue
                wave = math.ceil(math.ceil(N / max(1, 2 * sms // S)) / R) * 32
                for block in sorted({128, 256, min(512, max(32, wave))}):
                    out.append(KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U, stages=4))
    KB = math.ceil(K / 64)
    for rows in (128, 256) if M >= 32 else (128,):
        T = math.ceil(N / rows)
        Cs = [C for C in (1, 2, 4, 8, 16) if C <= KB and T * C <= 2 * sms]
        for C in sorted(Cs, reverse=True)[:2]:
            for P in (1, 2):
                out.append(KpCfg.make("tc05", split_k=C, rows=rows, k_unroll=2 if M <= 128 else 1,
                                      producers=P, stages=0))
    valid, seen = [], set()
    for c in out:
        key = tuple(getattr(c, f) for f, _ in c._fields_)
        if key in seen:
            continue
        seen.add(key)
        try:
            binding.scratch_bytes(M, N, K, c, sms)
            valid.append(c)
        except binding.KdaProjError:
            pass
    return valid


def _refuse_if_gave_up(what):
    """After a timing run: if a kernel wait ran out during it (the error word
    is set), report it and raise, so the candidate is dropped. Reading the word
    clears it, so the entry points accept the next candidate's calls."""
    torch.cuda.synchronize()
    code = binding.device_error()
    if code:
        what = what.as_dict() if isinstance(what, KpCfg) else what
        print(f"  a kernel wait ran out (code {code}) while timing {what}", file=sys.stderr)
        raise binding.KdaProjError(binding.KP_EDEVICE, f"kernel wait ran out (code {code})")


def sweep_shape(M, N, K, sms, device, kinds, verbose=False, quick=False):
    b = Bench(M, N, K, device)
    results = []
    cands = sweep_candidates(M, N, K, sms) if quick else candidates(M, N, K, sms, kinds)
    for c in cands:
        try:
            us = b.time_cfg(c, reps=5) if quick else b.time_cfg(c)
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


class PlanBench:
    """Full KDA projection timing: a weight stack of packed [N_qkvg+N_fab, K]
    + W_fb [N_fb, 128] layers (at least 4x L2 and at least 48, the layer count
    of the benchmark: each graph replay boundary breaks the chain of
    programmatic dependent launches, so short graphs favour the wrong mode),
    graph of `layers` calls."""

    def __init__(self, max_M, device, K=7168, Nq=4096, Nfab=136, Nfb=1024, seed=0):
        self.K, self.Nq, self.Nfab, self.Nfb = K, Nq, Nfab, Nfb
        per = ((Nq + Nfab) * K + Nfb * 128) * 2
        self.layers = max(48, math.ceil(4 * L2_BYTES / per))
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.Wp = (torch.randn((self.layers, Nq + Nfab, K), generator=g, device=device) * 0.02).to(torch.bfloat16)
        self.Wfb = (torch.randn((self.layers, Nfb, 128), generator=g, device=device) * 0.02).to(torch.bfloat16)
        self.device = device
        self.plan = binding.KdaPlan(K, Nq, Nfab, Nfb, max_M=max_M)
        self.stream = torch.cuda.Stream(device=device)
        self.aux = torch.cuda.Stream(device=device)
        with torch.cuda.stream(self.stream):
            self.evs = binding.make_events()

    def time_call(self, M, mode, reps=10, trials=3):
        """us per projection call at M tokens with the plan's current configs;
        mode 1 = overlapped, 0 = sequential."""
        x = torch.randn((M, self.K), device=self.device).to(torch.bfloat16)
        outs = self.plan.outputs(M, self.device)
        self.plan.set_overlap(mode)
        try:
            with torch.cuda.stream(self.stream):
                self.plan.run(x, self.Wp[0], self.Wfb[0], *outs, aux_stream=self.aux, events=self.evs)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for l in range(self.layers):
                    self.plan.run(x, self.Wp[l], self.Wfb[l], *outs, aux_stream=self.aux,
                                  events=self.evs)
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
            _refuse_if_gave_up(f"projection M={M} mode {mode}")
            return statistics.median(res)
        finally:
            self.plan.set_overlap(-1)


def tune_plan(ms, sms, device, verbose=False, top_q=3, top_b=2):
    """Joint choice per M of the Q/K/V/G, F_A/beta and F_B configurations that
    minimise the overlapped projection (the aux branch must co-run with the
    main one), and the per-M overlap flag (overlapped vs sequential with the
    same configurations)."""
    pb = PlanBench(max(ms), device)
    lines, dump = [], []
    for M in ms:
        q_res = sweep_shape(M, pb.Nq, pb.K, sms, device, ("cc", "tc05"))[:top_q]
        b_res = sweep_shape(M, pb.Nfb, 128, sms, device, ("cc", "tc05", "smallk"))[:top_b]
        f_cands = []
        for rows in (128, 256):
            for C in (1, 2, 4, 8, 16):
                for nkb in (1, 2, 4):
                    for stages in (2, 3):
                        for fuse in (0, binding.FLAG_FUSE_FB):
                            f_cands.append(KpCfg.make("tc05", split_k=C, rows=rows, k_unroll=nkb,
                                                      stages=stages, flags=binding.FLAG_PDL | fuse))
        if M <= 16:
            f_cands += [c for c in cc_candidates(M, pb.Nfab, pb.K, sms) if c.split_k <= 8]
        best = None
        skipped = []
        combos = []
        for (_, cq), cf in itertools.product(q_res, f_cands):
            # a fused F_A/beta launch computes F_B itself: one F_B candidate is enough
            for (_, cb) in (b_res[:1] if cf.flags & binding.FLAG_FUSE_FB else b_res):
                combos.append((cq, cb, cf))
        for cq, cb, cf in combos:
            try:
                plain = KpCfg.from_buffer_copy(cf)
                plain.flags &= ~binding.FLAG_FUSE_FB
                binding.scratch_bytes(M, pb.Nfab, pb.K, plain, sms)
                pb.plan.set_config(binding.BRANCH_QKVG, M, cq)
                pb.plan.set_config(binding.BRANCH_FAB, M, cf)
                pb.plan.set_config(binding.BRANCH_FB, M, cb)
                us = pb.time_call(M, 1)
            except binding.KdaProjError as e:
                skipped.append(e)
                if verbose:
                    print(f"  skip {cf.as_dict()}: {e}", file=sys.stderr)
                continue
            if verbose:
                print(f"  M={M} overlapped {us:8.3f} us  q={cq.as_dict()} f={cf.as_dict()} b={cb.as_dict()}",
                      file=sys.stderr)
            if best is None or us < best[0]:
                best = (us, cq, cf, cb)
        if best is None:
            raise RuntimeError(
                f"M={M}: no configuration combination ran ({len(q_res)} Q/K/V/G, {len(b_res)} F_B "
                f"and {len(f_cands)} F_A/beta candidates, {len(skipped)} refused"
                + (f"; first refusal: {skipped[0]}" if skipped else "") + ")")
        us_ovl, cq, cf, cb = best
        pb.plan.set_config(binding.BRANCH_QKVG, M, cq)
        pb.plan.set_config(binding.BRANCH_FAB, M, cf)
        pb.plan.set_config(binding.BRANCH_FB, M, cb)
        us_ovl = pb.time_call(M, 1)
        us_seq = pb.time_call(M, 0)
        # single launch over the packed weight: the best tcgen05 configs, and at
        # M <= 8 the CUDA-core kernel with one K slice (its F_A rows a cluster)
        us_one, c_one = None, None
        one_cands = [c for _, c in q_res if c.kind == binding.KIND_TC05] + tc05_candidates(
            M, pb.Nq + pb.Nfab, pb.K, sms)
        if M <= 8:
            one_cands += [KpCfg.make("cc", split_k=1, block=b, rows=R, k_unroll=U)
                          for (R, U) in ((1, 4), (2, 2), (2, 4), (4, 1), (4, 2))
                          for b in (128, 256, 512) if (b // 32) * R <= 128]
        for cand in one_cands:
            try:
                pb.plan.set_config(binding.BRANCH_QKVG, M, cand)
                us = pb.time_call(M, 2)
            except binding.KdaProjError:
                continue
            if verbose:
                print(f"  M={M} single launch {us:8.3f} us  {cand.as_dict()}", file=sys.stderr)
            if us_one is None or us < us_one:
                us_one, c_one = us, cand
        # decide between the modes on longer re-measurements (single runs of
        # 9-layer graphs differ by a few percent)
        pb.plan.set_config(binding.BRANCH_QKVG, M, cq)
        times = {0: pb.time_call(M, 0, reps=30, trials=5), 1: pb.time_call(M, 1, reps=30, trials=5)}
        if us_one is not None:
            pb.plan.set_config(binding.BRANCH_QKVG, M, c_one)
            times[2] = pb.time_call(M, 2, reps=30, trials=5)
            pb.plan.set_config(binding.BRANCH_QKVG, M, cq)
        us_seq, us_ovl = times[0], times[1]
        us_one = times.get(2)
        ov = min(times, key=times.get)
        if ov == 2:
            cq = c_one
            # The table holds one Q/K/V/G configuration per M, which the
            # two-stream mode then also runs: re-tune the aux branch for the
            # overlapped mode beside it, so that mode is tuned as well.
            pb.plan.set_config(binding.BRANCH_QKVG, M, cq)
            best_aux = None
            for cf2 in f_cands:
                for (_, cb2) in (b_res[:1] if cf2.flags & binding.FLAG_FUSE_FB else b_res):
                    try:
                        plain = KpCfg.from_buffer_copy(cf2)
                        plain.flags &= ~binding.FLAG_FUSE_FB
                        binding.scratch_bytes(M, pb.Nfab, pb.K, plain, sms)
                        pb.plan.set_config(binding.BRANCH_FAB, M, cf2)
                        pb.plan.set_config(binding.BRANCH_FB, M, cb2)
                        us = pb.time_call(M, 1)
                    except binding.KdaProjError:
                        continue
                    if best_aux is None or us < best_aux[0]:
                        best_aux = (us, cf2, cb2)
            if best_aux is not None:
                _, cf, cb = best_aux
                pb.plan.set_config(binding.BRANCH_FAB, M, cf)
                pb.plan.set_config(binding.BRANCH_FB, M, cb)
                times[1] = pb.time_call(M, 1, reps=30, trials=5)
                us_ovl = times[1]
                # the re-tuned two-stream mode may now beat the single launch
                ov = min(times, key=times.get)
        pb.plan.set_config(binding.BRANCH_QKVG, M, cq)
        lines += [table_line(M, pb.Nq, pb.K, cq, ov, times[ov]),
                  table_line(M, pb.Nfab, pb.K, cf, ov),
                  table_line(M, pb.Nfb, 128, cb, ov)]
        dump.append({"M": M, "overlapped_us": us_ovl, "sequential_us": us_seq,
                     "single_launch_us": us_one, "mode": ov,
                     "qkvg": cq.as_dict(), "fab": cf.as_dict(), "fb": cb.as_dict()})
        print(f"# M={M}: overlapped {us_ovl:.3f} us, sequential {us_seq:.3f} us, single launch "
              f"{us_one} us -> mode {ov}", flush=True)
        for l in lines[-3:]:
            print(l, flush=True)
    pb.plan.close()
    return lines, dump


def table_line(M, N, K, cfg, overlap=1, us=None):
    kind = binding.KIND_NAMES[cfg.kind]
    s = (f"{M} {N} {K} {kind} {cfg.split_k} {cfg.block} {cfg.rows} {cfg.k_unroll} {cfg.producers} "
         f"{cfg.stages} {cfg.flags} {overlap}")
    return s + (f"  # {us:.3f} us" if us is not None else "")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--shapes", default="kda",
                    help="kda-plan (joint, for the projection) | kda | sweep | N:K[,N:K...]")
    ap.add_argument("--m", type=int, nargs="*", default=None)
    ap.add_argument("--kinds", default="cc,tc05,smallk")
    ap.add_argument("--out", default=None)
    ap.add_argument("--json", default=None)
    ap.add_argument("--top", type=int, default=3)
    ap.add_argument("--append-to", default=None,
                    help="sweep: replace this table's lines for the swept (N, K) pairs with the "
                         "new ones and write it back")
    ap.add_argument("--full", action="store_true",
                    help="sweep: time the full candidate list instead of the short one")
    ap.add_argument("-v", action="store_true")
    args = ap.parse_args(argv)

    from .build import build
    build()
    binding.load()
    binding.table_clear()
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if args.shapes == "kda-plan":
        ms = args.m or [1, 2, 4, 8, 16, 32, 64, 128]
        lines, dump = tune_plan(ms, sms, dev, args.v)
        _write(args, dev, sms, lines, dump)
        return
    if args.shapes == "kda":
        shapes = KDA_SHAPES
        ms = args.m or [1, 2, 4, 8, 16, 32, 64, 128]
    elif args.shapes == "sweep":
        # the projection plan's own (N, K) pairs keep its jointly tuned entries
        shapes = [(n, k) for n in SWEEP_N for k in SWEEP_K if (n, k) not in KDA_SHAPES]
        ms = args.m or SWEEP_M
    else:
        shapes = [tuple(int(v) for v in s.split(":")) for s in args.shapes.split(",")]
        ms = args.m or [1, 2, 4, 8, 16, 32, 64, 128]
    kinds = tuple(args.kinds.split(","))
    lines, dump = [], []
    t0 = time.time()
    for (N, K) in shapes:
        for M in ms:
            res = sweep_shape(M, N, K, sms, dev, kinds, args.v,
                              quick=args.shapes == "sweep" and not args.full)
            if not res:
                continue
            best_us, best = res[0]
            lines.append(table_line(M, N, K, best, 1, best_us))
            dump.append({"M": M, "N": N, "K": K,
                         "results": [{"us": us, **c.as_dict()} for us, c in res[:args.top]]})
            print(lines[-1], flush=True)
    print(f"# sweep took {time.time() - t0:.1f} s", file=sys.stderr)
    _write(args, dev, sms, lines, dump)
    if args.append_to:
        swept = set(shapes)
        keep = []
        for line in open(args.append_to):
            if line.startswith("# shape sweep"):
                continue   # replaced by the new sweep's header below
            f = line.split("#")[0].split()
            if len(f) >= 3 and (int(f[1]), int(f[2])) in swept:
                continue
            keep.append(line.rstrip("\n"))
        with open(args.append_to, "w") as fh:
            fh.write("\n".join(keep + [f"# shape sweep ({len(lines)} entries, "
                                       f"{torch.cuda.get_device_name(dev)})"] + lines) + "\n")


def _write(args, dev, sms, lines, dump):
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
