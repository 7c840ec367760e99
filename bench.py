#!/usr/bin/env python3
"""Benchmark: Kimi-K3 KDA decode input projection on one GB300.

Workload: the full overlapped projection of one TP8 rank -- packed
[4096 + 136, 7168] bf16 weight (Q/K/V/G rows, then F_A/beta rows) and
W_fb [1024, 128] -- for token counts M in {1, 2, 4, 8, 16, 32, 64, 128}. Each
call reads a different layer of a 48-layer weight stack (2.92 GB, far above
the 129 MB L2) so weight reads come from HBM; x stays resident as in decode.

One step = one replay of a captured CUDA graph per M, each graph holding 48
projection calls (layers 0..47) = 384 calls. Reported value: mean over the M
values of the device time per call (us), median-free (total time / calls).

Also reported: per-M us/call, HBM GB/s and roofline fraction (bytes =
2(MK + NK + MN) summed over the three GEMMs), sequential vs overlapped times,
the dominant kernel's roofline (Q/K/V/G GEMM timed alone), the CPU oracle on
the host cores, the end-to-end number through host buffers, SM clocks, and
skinny_gemm_ex (fp16 inputs, residual add) at the Q/K/V/G shape.

--impl reference times the CPU oracle (the plain double-precision reference)
on a bounded column sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M_LIST = (1, 2, 4, 8, 16, 32, 64, 128)
K, N_QKVG, N_FAB, N_FA, N_FB = 7168, 4096, 136, 128, 1024
LAYERS = 48
METRIC = "KDA proj µs/call and HBM GB/s (% of ~8 TB/s) at M=1..128, bf16, 1×GB300"
UNIT = "us/call"
WORKLOAD = ("full KDA decode projection: packed [4096+136, 7168] bf16 + W_fb [1024,128] bf16; "
            "QKVG || F_A/beta->F_B (per-M mode from the table: two-stream overlap or one launch), "
            "graph-replayed, 48-layer weight stack rotated per call")


# ncu DRAM traffic of the single-launch projection kernels per token count (a
# profiles/ summary); used only while the kernels' sources are unchanged since
# that capture (their hash is recorded in it)
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "single_launch_n4232_k7168_dram_by_m.md")
KERNEL_SOURCES = [os.path.join(ROOT, "decode_projection_gemms_gb300", "csrc", f)
                  for f in ("kp_tc05.cu", "kp_cc_kernel.cuh", "kp_internal.cuh")]


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def load_traffic():
    """{M: DRAM bytes read + written per launch} from the summary, or None if
    it is missing or was taken on other kernel sources."""
    try:
        text = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None, "no ncu summary"
    import re
    m = re.search(r"kernel sources sha256\[:16\]: `?([0-9a-f]{16})", text)
    if not m or m.group(1) != kernel_source_hash():
        return None, "kernel sources changed since the ncu capture"
    rows = re.findall(r"^\|\s*(\d+)\s*\|\s*([\d.]+)\s*\|\s*([\d.]+)\s*\|", text, re.M)
    return {int(M): float(r) + float(w) for M, r, w in rows}, "ncu capture, " + os.path.relpath(
        TRAFFIC_SUMMARY, ROOT)


def call_bytes(M: int) -> int:
    """Algorithmic bytes of one projection call: 2(MK + NK + MN) per GEMM."""
    g = lambda m, n, k: 2 * (m * k + n * k + m * n)
    return g(M, N_QKVG, K) + g(M, N_FAB, K) + g(M, N_FB, N_FA)


def call_flops(M: int) -> int:
    return 2 * M * (N_QKVG * K + N_FAB * K + N_FB * N_FA)


def qkvg_bytes(M: int) -> int:
    return 2 * (M * K + N_QKVG * K + M * N_QKVG)


def load_peaks(burst: bool = False):
    """(HBM GB/s, bf16 TFLOP/s, source): the sustained tensor figure for the
    long decode step, the burst one for a kernel timed alone."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        tc = d["bf16_tflops"] if burst else d.get("bf16_tflops_sustained", d["bf16_tflops"])
        return float(d["hbm_gbs"]), float(tc), "measured"
    except Exception:
        return 6800.0, 1900.0 if burst else 1700.0, "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: each rank runs the same workload on its GPU)

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws):
    if ws <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group("gloo")
    return dist


def reduce_max(values, dist):
    """Element-wise max over ranks (host-side timing reduction, gloo)."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        if not shutil.which("nvidia-smi"):
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen(
            ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
             "--format=csv,noheader,nounits", "-lms", "100"],
            stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # samples under load: power above the idle floor
        pmax = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in loaded:
            for name, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": pmax}


# ---------------------------------------------------------------------------
# our arm

def run_ours(args):
    import torch
    from decode_projection_gemms_gb300 import binding
    from decode_projection_gemms_gb300.build import build
    from decode_projection_gemms_gb300.inputs import gen_kda_layer, gen_x

    ws, rank, local = dist_env()
    dist = dist_init(ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or ws == 1:
        build()
    barrier(dist)
    binding.load()
    hbm_peak, tc_peak, peak_src = load_peaks()
    tc_peak_burst = load_peaks(burst=True)[1]
    m_list = args.m or [m for m in M_LIST if m <= args.max_m]
    L = args.layers

    # weights: layer 0 from the canonical CPU stream, the rest drawn on the GPU
    wp_stack = torch.empty((L, N_QKVG + N_FAB, K), dtype=torch.bfloat16, device=dev)
    wfb_stack = torch.empty((L, N_FB, N_FA), dtype=torch.bfloat16, device=dev)
    for layer in range(L):
        wp, wfb = gen_kda_layer(layer, seed=0, device="cpu" if layer == 0 else dev)
        wp_stack[layer].copy_(wp)
        wfb_stack[layer].copy_(wfb)
        del wp, wfb
    xs = {M: gen_x(M, K, seed=0).to(dev) for M in m_list}
    outs = {M: (torch.empty((M, N_QKVG), dtype=torch.bfloat16, device=dev),
                torch.empty((M, N_FAB), dtype=torch.bfloat16, device=dev),
                torch.empty((M, N_FB), dtype=torch.bfloat16, device=dev)) for M in m_list}

    plan = binding.KdaPlan(K, N_QKVG, N_FAB, N_FB, max_M=max(max(m_list), 128))
    main = torch.cuda.Stream(device=dev)
    aux = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(main):
        evs = binding.make_events()

    def capture(M, mode, qkvg_only=False):
        plan.set_overlap(mode)
        g = torch.cuda.CUDAGraph()
        oq, of, ob = outs[M]
        # warm-up outside capture (lazy attribute setup)
        with torch.cuda.stream(main):
            if qkvg_only:
                binding.skinny_gemm(xs[M], wp_stack[0, :N_QKVG], oq,
                                    cfg=plan.get_config(binding.BRANCH_QKVG, M))
            else:
                plan.run(xs[M], wp_stack[0], wfb_stack[0], oq, of, ob, aux_stream=aux, events=evs)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=main):
            for layer in range(L):
                if qkvg_only:
                    binding.skinny_gemm(xs[M], wp_stack[layer, :N_QKVG], oq,
                                        cfg=plan.get_config(binding.BRANCH_QKVG, M))
                else:
                    plan.run(xs[M], wp_stack[layer], wfb_stack[layer], oq, of, ob,
                             aux_stream=aux, events=evs)
        plan.set_overlap(-1)
        return g

    graphs = {M: capture(M, -1) for M in m_list}
    graphs_seq = {M: capture(M, 0) for M in m_list}
    graphs_ovl = {M: capture(M, 1) for M in m_list}
    graphs_one = {M: capture(M, 2) for M in m_list}
    graphs_q = {M: capture(M, -1, qkvg_only=True) for M in m_list}

    def timed(gs, steps):
        """Replay each graph once per step; per-M device times (ms) summed.
        Events bracket every replay on the launching stream; no host sync
        inside the timed region."""
        ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in m_list] for _ in range(steps)]
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        e0.record(main)
        for s in range(steps):
            for i, M in enumerate(m_list):
                ev[s][i][0].record(main)
                gs[M].replay()
                ev[s][i][1].record(main)
        e1.record(main)
        torch.cuda.synchronize()
        barrier(dist)
        tot = {M: sum(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(steps))
               for i, M in enumerate(m_list)}
        return tot, e0.elapsed_time(e1)

    # warm-up
    with torch.cuda.stream(main):
        for _ in range(args.warmup):
            for M in m_list:
                graphs[M].replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(main):
        tot, wall_ms = timed(graphs, args.steps)
        tot_seq, _ = timed(graphs_seq, args.cmp_steps)
        tot_ovl, _ = timed(graphs_ovl, args.cmp_steps)
        tot_one, _ = timed(graphs_one, args.cmp_steps)
        tot_q, _ = timed(graphs_q, args.cmp_steps)
    e2e = run_e2e(args, plan, wp_stack, wfb_stack, m_list, dev, main, aux, evs, dist)
    ex = None if args.no_extras else run_ex(args, wp_stack, dev, main, hbm_peak, dist)
    cc = None if args.no_extras else run_cuda_core(args, wp_stack, dev, main, hbm_peak, dist)
    prefill = None if args.no_extras else run_prefill(args, wp_stack, dev, main, tc_peak_burst, dist)
    handoff = None if args.no_extras else run_handoff(args, plan, wp_stack, wfb_stack, xs, outs, dev,
                                                      main, aux, evs, dist)
    clock_info = clocks.stop()
    if cc is not None:
        # FP32-pipe roofline: 128 FMA lanes per SM at the highest SM clock seen
        mhz = clock_info.get("sm_max_mhz") or 2070.0
        alu_peak = torch.cuda.get_device_properties(dev).multi_processor_count * 128 * mhz * 1e6
        cc["alu_peak_fma_per_s"] = alu_peak
        for row in cc["per_m"].values():
            row["frac_of_alu_peak"] = round(row["fma_per_s"] / alu_peak, 4)
            row["fma_per_s"] = round(row["fma_per_s"], -6)

    # reductions (max over ranks)
    keys = list(m_list)
    vals = reduce_max([tot[M] for M in keys] + [tot_seq[M] for M in keys] +
                      [tot_ovl[M] for M in keys] + [tot_one[M] for M in keys] +
                      [tot_q[M] for M in keys] + [wall_ms], dist)
    nM = len(keys)
    tot = dict(zip(keys, vals[0:nM]))
    tot_seq = dict(zip(keys, vals[nM:2 * nM]))
    tot_ovl = dict(zip(keys, vals[2 * nM:3 * nM]))
    tot_one = dict(zip(keys, vals[3 * nM:4 * nM]))
    tot_q = dict(zip(keys, vals[4 * nM:5 * nM]))
    wall_ms = vals[5 * nM]

    per_m = {}
    for M in keys:
        us = tot[M] * 1e3 / (args.steps * L)
        us_seq = tot_seq[M] * 1e3 / (args.cmp_steps * L)
        us_ovl = tot_ovl[M] * 1e3 / (args.cmp_steps * L)
        us_one = tot_one[M] * 1e3 / (args.cmp_steps * L)
        us_q = tot_q[M] * 1e3 / (args.cmp_steps * L)
        roof_us = max(call_bytes(M) / (hbm_peak * 1e3), call_flops(M) / (tc_peak * 1e6))
        per_m[str(M)] = {
            "us_per_call": round(us, 3),
            "gbs": round(call_bytes(M) / (us * 1e3), 1),
            "roofline_us": round(roof_us, 3),
            "frac_of_roofline": round(roof_us / us, 4),
            "frac_of_8tbs": round(call_bytes(M) / (us * 1e3) / 8000.0, 4),
            "mode": {0: "sequential", 1: "overlapped", 2: "single-launch"}[plan.overlap_at(M)],
            "us_sequential": round(us_seq, 3),
            "us_overlapped": round(us_ovl, 3),
            "us_single_launch": round(us_one, 3),
            "overlap_speedup": round(us_seq / us_ovl, 4),
            "qkvg_kernel_us": round(us_q, 3),
            "qkvg_kernel_gbs": round(qkvg_bytes(M) / (us_q * 1e3), 1),
            "configs": {b: plan.get_config(i, M).as_dict()
                        for i, b in enumerate(("qkvg", "fab", "fb"))},
        }
    value = statistics.fmean(per_m[str(M)]["us_per_call"] for M in keys)
    # our kernel launches per projection call in the timed mode: one for the
    # single launch; Q/K/V/G + F_A/beta (+ F_B unless it is fused) otherwise
    def launches_per_call(M):
        if plan.overlap_at(M) == 2:
            return 1
        fused = plan.get_config(binding.BRANCH_FAB, M).flags & binding.FLAG_FUSE_FB
        return 2 if fused else 3
    q_bytes = sum(qkvg_bytes(M) for M in keys)
    q_time_us = sum(per_m[str(M)]["qkvg_kernel_us"] for M in keys)
    if cc is not None:
        for Ms, row in cc["per_m"].items():
            if Ms in per_m:   # the tcgen05 kernel on the same shape, same run
                row["tcgen05_us"] = per_m[Ms]["qkvg_kernel_us"]
    q_achieved = q_bytes / (q_time_us * 1e3)  # GB/s
    # The timed mode's dominant kernel: the single-launch projection where the
    # table picks it (one kernel per call), else the Q/K/V/G GEMM.
    for M in keys:
        row = per_m[str(M)]
        if plan.overlap_at(M) == 2:
            kind = binding.KIND_NAMES[plan.get_config(binding.BRANCH_QKVG, M).kind]
            row["timed_kernel"] = {"kernel": f"single-launch projection ({kind})",
                                   "us": row["us_single_launch"],
                                   "gbs": round(call_bytes(M) / (row["us_single_launch"] * 1e3), 1)}
        else:
            row["timed_kernel"] = {"kernel": "Q/K/V/G GEMM", "us": row["qkvg_kernel_us"],
                                   "gbs": row["qkvg_kernel_gbs"]}
        row["timed_kernel"]["frac_of_hbm"] = round(row["timed_kernel"]["gbs"] / hbm_peak, 4)
    one = [M for M in keys if plan.overlap_at(M) == 2]
    traffic, traffic_src = load_traffic()
    if one:
        o_bytes = sum(call_bytes(M) for M in one)
        o_time = sum(per_m[str(M)]["us_single_launch"] for M in one)
        tr = None
        if traffic is not None and all(M in traffic for M in one):
            tr = round(statistics.fmean(traffic[M] for M in one))
        roofline = {"bound": "hbm", "achieved": round(o_bytes / (o_time * 1e3), 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(o_bytes / (o_time * 1e3) / hbm_peak, 4),
                    "traffic": tr,
                    "algorithmic_bytes_per_launch": round(o_bytes / len(one)),
                    "traffic_source": traffic_src if tr is not None else
                    f"null: {traffic_src if traffic is None else 'capture lacks some M'}",
                    "kernel": "single-launch projection over the packed [4232, 7168] weight with "
                              "F_B fused (the timed mode's only kernel per call): CUDA-core at M "
                              f"{[M for M in one if plan.get_config(0, M).kind == binding.KIND_CC]}, "
                              "tcgen05 at M "
                              f"{[M for M in one if plan.get_config(0, M).kind == binding.KIND_TC05]}",
                    "M": one,
                    "units": "achieved = sum over these M of 2(MK+NK+MN) bytes of the three GEMMs / "
                             "sum of per-launch device time; traffic = mean DRAM read+write "
                             "bytes per launch over the same M",
                    "peak_source": f"{peak_src} hbm_gbs (copy bandwidth, burst)"}
    else:
        roofline = {"bound": "hbm", "achieved": round(q_achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(q_achieved / hbm_peak, 4), "traffic": None,
                    "kernel": "Q/K/V/G GEMM", "peak_source": f"{peak_src} hbm_gbs"}
    roofline_qkvg = {"achieved": round(q_achieved, 1), "unit": "GB/s",
                     "frac": round(q_achieved / hbm_peak, 4), "M": keys,
                     "kernel": "Q/K/V/G GEMM (per-M configured kernel), timed alone"}
    eager = None if args.no_extras else run_eager(args, plan, wp_stack, wfb_stack, xs, outs, main,
                                                  aux, evs, dist)
    n_launches = args.steps * L * sum(launches_per_call(M) for M in keys)
    cpu = run_cpu_baseline(args, m_list) if (rank == 0 and not args.no_cpu) else None
    plan.close()
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 3),
            "unit": UNIT,
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(wall_ms / args.steps, 4),
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded; x ~ N(0,1), W ~ N(0, 0.02^2); random weights)",
            "config": {"workload": WORKLOAD, "M": keys, "K": K, "N_qkvg": N_QKVG,
                       "N_fab": N_FAB, "N_fb": N_FB, "layers": L,
                       "weight_stack_gb": round(L * (N_QKVG + N_FAB) * K * 2 / 1e9 +
                                                L * N_FB * N_FA * 2 / 1e9, 3),
                       "l2": "inputs larger than L2: weight stack rotated per call",
                       "value_is": "mean over M of device time per projection call",
                       "parallelism": f"replicas x{ws}"},
            "per_m": per_m,
            "roofline": roofline,
            "roofline_qkvg_alone": roofline_qkvg,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": n_launches,
            "skinny_gemm_ex": ex,
            "cuda_core_splitk": cc,
            "prefill": prefill,
            "pdl_handoff": handoff,
            "eager": eager,
            "clocks": clock_info,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_ex(args, wp_stack, dev, main, hbm_peak, dist, m_ex=(1, 16)):
    """skinny_gemm_ex at the Q/K/V/G shape (N=4096, K=7168): bf16 and fp16
    inputs, with and without a residual, each as a graph of one call per
    layer of the rotated weight stack (device time per call)."""
    import torch
    from decode_projection_gemms_gb300 import binding
    from decode_projection_gemms_gb300.inputs import gen_x

    L = wp_stack.shape[0]
    stacks = {"bf16": wp_stack[:, :N_QKVG], "fp16": wp_stack[:, :N_QKVG].to(torch.float16)}
    out = {"shape": {"N": N_QKVG, "K": K}, "layers": L, "per_m": {}}
    for M in m_ex:
        row = {}
        for dt, tdt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
            x = gen_x(M, K, seed=0, dtype=tdt).to(dev)
            r = gen_x(M, N_QKVG, seed=1, dtype=tdt).to(dev)
            y = torch.empty((M, N_QKVG), dtype=tdt, device=dev)
            for with_res in (False, True):
                res = r if with_res else None
                with torch.cuda.stream(main):
                    binding.skinny_gemm_ex(x, stacks[dt][0], res, y)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=main):
                    for layer in range(L):
                        binding.skinny_gemm_ex(x, stacks[dt][layer], res, y)
                with torch.cuda.stream(main):
                    g.replay()
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(main)
                    for _ in range(args.cmp_steps):
                        g.replay()
                    b.record(main)
                torch.cuda.synchronize()
                us = reduce_max([a.elapsed_time(b)], dist)[0] * 1e3 / (args.cmp_steps * L)
                nbytes = qkvg_bytes(M) + (M * N_QKVG * 2 if with_res else 0)
                key = dt + ("_residual" if with_res else "")
                row[key] = {"us_per_call": round(us, 3), "gbs": round(nbytes / (us * 1e3), 1),
                            "frac_of_roofline": round(nbytes / (us * 1e3) / hbm_peak, 4)}
        out["per_m"][str(M)] = row
    del stacks
    return out


def run_cuda_core(args, wp_stack, dev, main, hbm_peak, dist, m_cc=(1, 4, 8, 16)):
    """The CUDA-core split-K GEMV at the Q/K/V/G shape (N=4096, K=7168), the
    kernel kind the projection would use at M <= 16 without the tcgen05
    kernel: the fastest of its candidate configurations per M (short runs,
    then the winner re-timed), as a graph of one call per layer of the
    rotated weight stack. Reports the HBM fraction and the FMA rate (M*N*K
    fused multiply-adds per call) for the FP32-pipe roofline."""
    import torch
    from decode_projection_gemms_gb300 import binding
    from decode_projection_gemms_gb300.autotune import cc_candidates
    from decode_projection_gemms_gb300.inputs import gen_x

    L = wp_stack.shape[0]
    W = wp_stack[:, :N_QKVG]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"shape": {"N": N_QKVG, "K": K}, "layers": L, "per_m": {}}

    def time_cfg(x, y, cfg, reps):
        with torch.cuda.stream(main):
            binding.skinny_gemm(x, W[0], y, cfg=cfg)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            for layer in range(L):
                binding.skinny_gemm(x, W[layer], y, cfg=cfg)
        with torch.cuda.stream(main):
            g.replay()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(main)
            for _ in range(reps):
                g.replay()
            b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / (reps * L)

    for M in m_cc:
        x = gen_x(M, K, seed=3).to(dev)
        y = torch.empty((M, N_QKVG), dtype=torch.bfloat16, device=dev)
        best = None
        for cfg in cc_candidates(M, N_QKVG, K, sms):
            try:
                binding.scratch_bytes(M, N_QKVG, K, cfg, sms)
            except binding.KdaProjError:
                continue
            us = time_cfg(x, y, cfg, 2)
            if best is None or us < best[0]:
                best = (us, cfg)
        us = reduce_max([time_cfg(x, y, best[1], args.cmp_steps)], dist)[0]
        nbytes = qkvg_bytes(M)
        out["per_m"][str(M)] = {"us_per_call": round(us, 3), "gbs": round(nbytes / (us * 1e3), 1),
                                "frac_of_hbm_roofline": round(nbytes / (us * 1e3) / hbm_peak, 4),
                                "fma_per_s": M * N_QKVG * K / (us * 1e-6),
                                "config": best[1].as_dict()}
    return out


def run_prefill(args, wp_stack, dev, main, tc_peak, dist, m_pre=(256, 1024, 4096), layers=8):
    """skinny_gemm at prefill token counts on the Q/K/V/G weights (N=4096,
    K=7168): one tcgen05 launch per call with token tiles of 256 on the grid,
    against calling it once per 256-token slice (which streams the weights
    from HBM once per slice). Device time per call, TFLOP/s."""
    import torch
    from decode_projection_gemms_gb300 import binding
    from decode_projection_gemms_gb300.inputs import gen_x

    L = min(layers, wp_stack.shape[0])
    out = {"shape": {"N": N_QKVG, "K": K}, "layers": L, "per_m": {}}
    for M in m_pre:
        x = gen_x(M, K, seed=2).to(dev)
        y = torch.empty((M, N_QKVG), dtype=torch.bfloat16, device=dev)

        def call(layer, sliced):
            w = wp_stack[layer, :N_QKVG]
            if not sliced:
                binding.skinny_gemm(x, w, y)
            else:
                for m0 in range(0, M, 256):
                    binding.skinny_gemm(x[m0:m0 + 256], w, y[m0:m0 + 256])

        row = {}
        for sliced in (False, True):
            with torch.cuda.stream(main):
                call(0, sliced)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                for layer in range(L):
                    call(layer, sliced)
            reps = max(2, args.cmp_steps // 4)
            with torch.cuda.stream(main):
                g.replay()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(main)
                for _ in range(reps):
                    g.replay()
                b.record(main)
            torch.cuda.synchronize()
            us = reduce_max([a.elapsed_time(b)], dist)[0] * 1e3 / (reps * L)
            tf = 2.0 * M * N_QKVG * K / (us * 1e6)
            row["per_256_slices" if sliced else "one_launch"] = {
                "us_per_call": round(us, 2), "tflops": round(tf, 1),
                "frac_of_tensor_peak": round(tf / tc_peak, 4)}
        out["per_m"][str(M)] = row
    return out


def run_handoff(args, plan, wp_stack, wfb_stack, xs, outs, dev, main, aux, evs, dist, m_h=(1, 16)):
    """A downstream kernel after every projection call (it reads all of
    out_qkvg), launched with programmatic dependent launch or without: the
    difference is the part of its launch and prologue that overlaps the
    projection's tail. Device time per (projection + consumer) pair."""
    import torch
    from decode_projection_gemms_gb300 import binding
    L = args.layers
    acc = torch.zeros(1, dtype=torch.int64, device=dev)
    out = {"consumer": "reads out_qkvg (M x 4096 bf16) after griddepcontrol.wait", "per_m": {}}
    for M in m_h:
        if M not in xs:
            continue
        oq, of, ob = outs[M]
        row = {}
        for pdl in (True, False):
            def body():
                for layer in range(L):
                    plan.run(xs[M], wp_stack[layer], wfb_stack[layer], oq, of, ob,
                             aux_stream=aux, events=evs)
                    binding.pdl_consumer_checksum(oq, acc, pdl=pdl)
            with torch.cuda.stream(main):
                body()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=main):
                body()
            reps = max(2, args.cmp_steps // 2)
            with torch.cuda.stream(main):
                g.replay()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(main)
                for _ in range(reps):
                    g.replay()
                b.record(main)
            torch.cuda.synchronize()
            us = reduce_max([a.elapsed_time(b)], dist)[0] * 1e3 / (reps * L)
            row["pdl" if pdl else "no_pdl"] = round(us, 3)
        out["per_m"][str(M)] = row
    return out


def run_eager(args, plan, wp_stack, wfb_stack, xs, outs, main, aux, evs, dist, m_e=(1, 16, 128)):
    """The projection called eagerly (no graph): host time per call to enqueue
    it, through the Python binding and through the bare C ABI (ctypes with
    prepared arguments), and the device time per call of each eager chain of
    48 calls (one layer each); a chain whose host time per call exceeds the
    kernels' is paced by the host."""
    import ctypes
    import torch
    from decode_projection_gemms_gb300 import binding
    L = args.layers
    lib = binding.load()
    out = {"calls_per_sample": L, "per_m": {}}
    for M in m_e:
        if M not in xs:
            continue
        oq, of, ob = outs[M]
        ms = ctypes.c_void_p(int(main.cuda_stream))
        ax = ctypes.c_void_p(int(aux.cuda_stream))
        ev = (ctypes.c_void_p * 2)(int(evs[0].cuda_event), int(evs[1].cuda_event))
        h = ctypes.c_void_p(plan.handle)
        raw = [(h, ctypes.c_void_p(xs[M].data_ptr()), ctypes.c_void_p(wp_stack[layer].data_ptr()),
                ctypes.c_void_p(wfb_stack[layer].data_ptr()), ctypes.c_void_p(oq.data_ptr()),
                ctypes.c_void_p(of.data_ptr()), ctypes.c_void_p(ob.data_ptr()), M, ms, ax, ev)
               for layer in range(L)]
        host_py, host_c, dev_py, dev_c = [], [], [], []
        with torch.cuda.stream(main):
            for rep in range(6):
                torch.cuda.synchronize()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(main)
                t0 = time.perf_counter()
                if rep % 2 == 0:
                    for layer in range(L):
                        plan.run(xs[M], wp_stack[layer], wfb_stack[layer], oq, of, ob,
                                 aux_stream=aux, events=evs)
                else:
                    for r in raw:
                        if lib.kda_proj_run(*r) != 0:
                            raise binding.KdaProjError(-5, binding.last_error())
                t1 = time.perf_counter()
                b.record(main)
                torch.cuda.synchronize()
                if rep >= 2:   # the first pair warms up
                    (host_py if rep % 2 == 0 else host_c).append((t1 - t0) * 1e6 / L)
                    (dev_py if rep % 2 == 0 else dev_c).append(a.elapsed_time(b) * 1e3 / L)
        vals = reduce_max([statistics.median(host_py), statistics.median(host_c),
                           statistics.median(dev_py), statistics.median(dev_c)], dist)
        out["per_m"][str(M)] = {"host_us_per_call_binding": round(vals[0], 2),
                                "host_us_per_call_c_abi": round(vals[1], 2),
                                "device_us_per_call_eager_binding": round(vals[2], 3),
                                "device_us_per_call_eager_c_abi": round(vals[3], 3)}
    return out


def run_e2e(args, plan, wp_stack, wfb_stack, m_list, dev, main, aux, evs, dist):
    """Same metric through the public API with host buffers: every call has
    its own x in pinned host memory and its own output block (the three
    outputs are consecutive slices of one block), and every call's x goes to
    the device and its outputs come back inside the timed region. The calls
    run in chunks: a chunk's inputs go over in one copy on a side stream
    while the previous chunk computes, and its outputs come back in one copy
    on another side stream while the next chunk computes. Small M, where a
    copy's fixed cost dominates, takes the whole chain as one chunk."""
    import torch
    from decode_projection_gemms_gb300.inputs import gen_x
    L = args.layers
    NOUT = N_QKVG + N_FAB + N_FB
    cin = torch.cuda.Stream(device=dev)
    cout = torch.cuda.Stream(device=dev)
    hx = {M: gen_x(L * M, K, seed=M).view(L, M, K).pin_memory() for M in m_list}
    dx = {M: torch.empty((L, M, K), dtype=torch.bfloat16, device=dev) for M in m_list}
    dblk = {M: torch.empty((L, M * NOUT), dtype=torch.bfloat16, device=dev) for M in m_list}
    hblk = {M: torch.empty((L, M * NOUT), dtype=torch.bfloat16).pin_memory() for M in m_list}

    def chunk_of(M):
        return L if M <= 4 else min(L, 8)

    def outs(M, layer):
        flat = dblk[M][layer]
        a, b = M * N_QKVG, M * (N_QKVG + N_FAB)
        return (flat[:a].view(M, N_QKVG), flat[a:b].view(M, N_FAB), flat[b:].view(M, N_FB))

    def calls(M):
        CH = chunk_of(M)
        bounds = [(c, min(c + CH, L)) for c in range(0, L, CH)]
        ev_in = [torch.cuda.Event() for _ in bounds]
        ev_run = [torch.cuda.Event() for _ in bounds]
        start = torch.cuda.Event()
        start.record(main)
        cin.wait_event(start)
        cout.wait_event(start)
        with torch.cuda.stream(cin):
            for i, (a, b) in enumerate(bounds):
                dx[M][a:b].copy_(hx[M][a:b], non_blocking=True)
                ev_in[i].record(cin)
        for i, (a, b) in enumerate(bounds):
            main.wait_event(ev_in[i])
            for layer in range(a, b):
                plan.run(dx[M][layer], wp_stack[layer], wfb_stack[layer], *outs(M, layer),
                         aux_stream=aux, events=evs)
            ev_run[i].record(main)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_run[i])
                hblk[M][a:b].copy_(dblk[M][a:b], non_blocking=True)
        end = torch.cuda.Event()
        end.record(cout)
        main.wait_event(end)                              # join the copy streams

    graphs = {}
    for M in m_list:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(main):
            calls(M)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=main):
            calls(M)
        graphs[M] = g
    steps = max(1, args.cmp_steps)
    tot = {M: 0.0 for M in m_list}
    with torch.cuda.stream(main):
        for M in m_list:
            graphs[M].replay()
        torch.cuda.synchronize()
        barrier(dist)
        for _ in range(steps):
            for M in m_list:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(main)
                graphs[M].replay()
                b.record(main)
                b.synchronize()
                tot[M] += a.elapsed_time(b)
    # the host copy of the last call's outputs is what the device wrote
    for M in m_list:
        assert torch.equal(hblk[M][L - 1], dblk[M][L - 1].cpu()), f"e2e read-back mismatch at M={M}"
    vals = reduce_max([tot[M] for M in m_list], dist)
    us = [v * 1e3 / (steps * L) for v in vals]
    h2d = sum(M * K * 2 for M in m_list) * L
    d2h = sum(M * NOUT * 2 for M in m_list) * L
    return {"value": round(statistics.fmean(us), 3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "per_m_us": {str(M): round(u, 3) for M, u in zip(m_list, us)},
            "calls_per_copy": {str(M): chunk_of(M) for M in m_list}}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)

def oracle_step(stride: int, nthreads: int, m_list):
    """Oracle on a column sample (every `stride`-th output feature of each
    GEMM); returns host seconds per call, averaged over M, scaled back to the
    full column count."""
    import numpy as np
    import oracle
    from decode_projection_gemms_gb300.inputs import bf16_bits, gen_kda_layer, gen_x
    wp, wfb = gen_kda_layer(0, seed=0)
    wpb, wfbb = bf16_bits(wp), bf16_bits(wfb)
    wq = np.ascontiguousarray(wpb[:N_QKVG:stride])
    wf = wpb[N_QKVG:]
    wfs = np.ascontiguousarray(wfbb[::stride])
    times = []
    for M in m_list:
        xb = bf16_bits(gen_x(M, K, seed=0))
        t0 = time.perf_counter()
        oracle.gemm(xb, wq, nthreads)
        fab = oracle.gemm(xb, wf, nthreads)               # F_A/beta is small: all columns
        fa = oracle.f64_to_bf16(fab[:, :N_FA])
        oracle.gemm(fa, wfs, nthreads)
        dt = time.perf_counter() - t0
        # scale the sampled Q/K/V/G and F_B parts to all columns
        frac_sampled = (wq.shape[0] * K + N_FAB * K + wfs.shape[0] * N_FA)
        frac_full = (N_QKVG * K + N_FAB * K + N_FB * N_FA)
        times.append(dt * frac_full / frac_sampled)
    return statistics.fmean(times)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(line.split(":", 1) for line in out.splitlines() if ":" in line)
        fields = {k.strip(): v.strip() for k, v in fields.items()}
        name = fields.get("Model name")
        if name:
            vendor = fields.get("Vendor ID")
            return f"{vendor} {name}" if vendor and vendor not in name else name
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def run_cpu_baseline(args, m_list):
    """The oracle on the host: all cores over output features (all columns),
    and one thread on a column sample (every 16th feature, scaled up)."""
    nthreads = os.cpu_count() or 1
    t = oracle_step(1, nthreads, m_list)
    t1 = oracle_step(16, 1, m_list)
    return {"value": round(t * 1e6, 1), "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"double-precision oracle, full projection (all output features), one "
                      f"call per M in {list(m_list)} on layer 0, {nthreads} threads over output "
                      f"features; mean over M",
            "single_thread": {"value": round(t1 * 1e6, 1), "unit": UNIT, "cores": 1,
                              "sample": "one thread, every 16th output feature of Q/K/V/G and "
                                        "F_B (all of F_A/beta), scaled to all features; mean "
                                        "over the same M values"}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    m_list = args.m or [m for m in M_LIST if m <= args.max_m]
    nthreads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_step(args.cpu_stride * 4, nthreads, m_list[:1])
    t0 = time.perf_counter()
    vals = [oracle_step(args.cpu_stride, nthreads, m_list) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    value = statistics.fmean(vals) * 1e6
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall * 1e3 / max(1, args.steps), 2),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; x ~ N(0,1), W ~ N(0, 0.02^2))",
        "config": {"workload": WORKLOAD, "M": m_list, "K": K, "N_qkvg": N_QKVG, "N_fab": N_FAB,
                   "N_fb": N_FB, "value_is": "mean over M of host time per projection call"},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": nthreads,
                         "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": f"every {args.cpu_stride}th output feature of Q/K/V/G and F_B, "
                                   "all of F_A/beta, scaled to all columns"},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--max-m", type=int, default=128)
    ap.add_argument("--m", type=int, nargs="*", default=None,
                    help="token counts to run (default 1 2 4 ... 128 up to --max-m)")
    ap.add_argument("--cmp-steps", type=int, default=20,
                    help="steps for the sequential/overlapped/kernel-alone comparisons")
    ap.add_argument("--cpu-stride", type=int, default=16,
                    help="column sampling stride of the CPU oracle")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the skinny_gemm_ex and prefill measurements (e.g. for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
