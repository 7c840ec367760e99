"""Shared helpers for the GPU parity tests (inputs from the seeded generators,
expected values from the CPU oracle only)."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.inputs import bf16_bits, gen_kda_layer, gen_w, gen_x

NTHREADS = os.cpu_count() or 1
NAN_BF16 = float("nan")


def poisoned(shape, device="cuda"):
    """Output buffer pre-filled with NaN, so any element a kernel skips fails."""
    return torch.full(shape, NAN_BF16, dtype=torch.bfloat16, device=device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def gemm_case(M, N, K, seed=0, dist="normal"):
    x = gen_x(M, K, seed=seed, dist=dist)
    W = gen_w(N, K, seed=seed + 1)
    return x, W


def check_gemm(x, W, cfg=None, label=""):
    M, K = x.shape
    N = W.shape[0]
    y = poisoned((M, N))
    binding.skinny_gemm(x.cuda(), W.cuda(), y, cfg=cfg)
    torch.cuda.synchronize()
    ref = oracle.gemm(bf16_bits(x), bf16_bits(W), nthreads=NTHREADS)
    r = oracle.compare(to_f64(y), ref)
    assert r["ok"], f"{label} M={M} N={N} K={K} cfg={cfg.as_dict() if cfg else 'auto'}: {r}"
    return y, r


def kda_reference(x, wp, wfb, n_qkvg, n_fab):
    """Oracle outputs plus the a-priori bound for F_B computed from the
    oracle's F_A: F_A itself may differ from the GPU's by its own tolerance,
    which propagates through W_fb."""
    qkvg, fab, fa_bits, fb = oracle.kda_proj(bf16_bits(x), bf16_bits(wp), bf16_bits(wfb),
                                             n_qkvg, n_fab, 128, nthreads=NTHREADS)
    fa = oracle.bf16_to_f64(fa_bits)
    dfa = oracle.tolerance(fab[:, :128]) + oracle.ulp_bf16(fa)       # |F_A gpu - F_A ref| bound
    wfb_abs = np.abs(oracle.bf16_to_f64(bf16_bits(wfb)))
    fb_extra = dfa @ wfb_abs.T
    return qkvg, fab, fb, fb_extra


def check_fb_stage(out_fab, out_fb, wfb, label=""):
    """F_B checked on its own: the oracle's F_B computed from the GPU's own bf16
    F_A (columns 0..127 of out_fab), against out_fb at the plain bound
    4 ulp_bf16(|ref|) + 1e-3 with nothing added. F_B's input is the bf16 F_A
    output, read in place ("[Kimi-K3] Overlap low-M TP8 KDA projections",
    section 关键源码片段, run_fab_fb)."""
    fa_gpu = bf16_bits(out_fab[:, :128].contiguous().cpu())
    ref = oracle.gemm(fa_gpu, bf16_bits(wfb.cpu()), nthreads=NTHREADS)
    r = oracle.compare(to_f64(out_fb), ref)
    assert r["ok"], f"{label} fb (stage-isolated, from the GPU's F_A): {r}"
    return r


def check_kda(outs, x, wp, wfb, n_qkvg, n_fab, label="", ref=None):
    """All three outputs against the oracle. F_B twice: end to end from the
    oracle's own F_A (bound widened by the propagated F_A tolerance), and
    stage-isolated from the GPU's F_A at the plain bound. ``ref``: a
    kda_reference() result for these inputs, to reuse across calls."""
    oq, of, ob = outs
    qkvg, fab, fb, fb_extra = ref if ref is not None else kda_reference(x, wp, wfb, n_qkvg, n_fab)
    for name, got, ref, extra in (("qkvg", oq, qkvg, None), ("fab", of, fab, None),
                                  ("fb", ob, fb, fb_extra)):
        r = oracle.compare(to_f64(got), ref, extra=extra)
        assert r["ok"], f"{label} {name}: {r}"
    check_fb_stage(of, ob, wfb, label)


def kda_inputs(M, layer=0, seed=0, K=7168, Nq=4096, Nfab=136, Nfb=1024):
    x = gen_x(M, K, seed=seed)
    wp, wfb = gen_kda_layer(layer, seed=seed, K=K, N_qkvg=Nq, N_fab=Nfab, N_fb=Nfb)
    return x, wp, wfb
