"""Pins for the CPU oracle: facts fixed by the mathematics, not by the oracle.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with something that the definition ``y = x * W^T`` (skinny
GEMM docstring of the Kimi K3 support page, part 1 (vllm PR #50089 digest,
CuteSkinnyGemm) and the
chained projection of "[Kimi-K3] Overlap low-M TP8 KDA projections"
(run_kda_projection_overlap) fix independently:

* hand-derived bf16 rounding cases (``golden/bf16_rne_cases.txt``);
* exact bf16 widening, checked against a bit-field decode written here;
* closed forms: all-ones gives exactly K; a one-hot row selects a column of W;
  a chain whose intermediate F_A needs rounding gives a hand-computed value;
* invariants: power-of-two scaling, row independence, thread-count
  independence, the packed weight's row slices;
* brute force: exact rational sums on tiny shapes, against which the double
  oracle must sit within the summation error bound.

The same page's kernel also takes fp16 inputs and adds an optional residual
after the K loop (C = A * B^T + residual); ``gemm_ex`` is pinned by
hand-derived fp16 decodings (``golden/fp16_decode_cases.txt``), an exact
bit-field decode, closed forms with a residual and rational brute force.

``test_oracle_mutants.py`` runs every pin against deliberately broken copies
of the oracle's C source to show each plausible mistake trips at least one.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

from decode_projection_gemms_gb300.inputs import bf16_bits, bits16, gen_w, gen_x

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bf16_exact(bits: int) -> Fraction:
    """Exact value of a (finite) bf16 bit pattern, from its bit fields."""
    s = (bits >> 15) & 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    assert e != 0xFF, "not finite"
    if e == 0:
        v = Fraction(f, 1 << 133)
    else:
        v = Fraction(128 + f, 128) * (Fraction(2) ** (e - 127))
    return -v if s else v


def fp16_exact(bits: int) -> Fraction:
    """Exact value of a (finite) fp16 bit pattern, from its bit fields."""
    s = (bits >> 15) & 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    assert e != 0x1F, "not finite"
    if e == 0:
        v = Fraction(f, 1 << 24)
    else:
        v = Fraction(1024 + f, 1024) * (Fraction(2) ** (e - 15))
    return -v if s else v


def load_fp16_cases():
    cases = []
    with open(os.path.join(GOLDEN, "fp16_decode_cases.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            v = {"inf": float("inf"), "-inf": float("-inf"), "nan": float("nan")}.get(parts[1])
            cases.append((int(parts[0], 16), float.fromhex(parts[1]) if v is None else v, line))
    return cases


def load_rne_cases():
    cases = []
    with open(os.path.join(GOLDEN, "bf16_rne_cases.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            cases.append((float.fromhex(parts[0]), int(parts[1], 16), line))
    return cases


def _bits(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t)


def _const_bf16(shape, value: float) -> np.ndarray:
    t = torch.full(shape, value, dtype=torch.float32).to(torch.bfloat16)
    assert float(t.flatten()[0]) == value, "constant must be exact in bf16"
    return _bits(t)


def _const(shape, value: float, dtype: str) -> np.ndarray:
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    t = torch.full(shape, value, dtype=torch.float32).to(tdt)
    assert float(t.flatten()[0]) == value, f"constant must be exact in {dtype}"
    return bits16(t)


def _exact(bits: int, dtype: str) -> Fraction:
    return bf16_exact(bits) if dtype == "bf16" else fp16_exact(bits)


# ---- pins ---------------------------------------------------------------------

def pin_rne_golden(orc):
    cases = load_rne_cases()
    vals = np.array([c[0] for c in cases], dtype=np.float64)
    got = orc.f64_to_bf16(vals)
    for (v, want, line), g in zip(cases, got):
        assert int(g) == want, f"bf16({v!r}) = {int(g):04X}, want {want:04X}  [{line}]"


def pin_widen_exact(orc):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint32).astype(np.uint16)
    finite = ((bits >> 7) & 0xFF) != 0xFF
    bits = bits[finite]
    got = orc.bf16_to_f64(bits)
    for b, g in zip(bits.tolist(), got.tolist()):
        assert Fraction(g) == bf16_exact(b), f"widen({b:04X}) = {g!r}"


def pin_all_ones(orc):
    # every partial sum is an integer <= 2^24, so y = K exactly
    for K in (1, 128, 1024, 2048, 7168, 16384):
        x = _const_bf16((2, K), 1.0)
        w = _const_bf16((3, K), 1.0)
        y = orc.gemm(x, w)
        assert np.array_equal(y, np.full((2, 3), float(K))), f"K={K}: {y}"


def pin_one_hot(orc):
    M, K, N = 4, 64, 24
    w = _bits(gen_w(N, K, seed=11, std=1.0))
    cols = [0, 5, 63, 17]
    xf = torch.zeros(M, K)
    for m, j in enumerate(cols):
        xf[m, j] = 1.0
    y = orc.gemm(_bits(xf.to(torch.bfloat16)), w)
    for m, j in enumerate(cols):
        for n in range(N):
            want = bf16_exact(int(w[n, j]))
            assert Fraction(float(y[m, n])) == want, f"y[{m},{n}] != W[{n},{j}]"


def pin_pow2_scaling(orc):
    x = gen_x(3, 96, seed=3)
    w = _bits(gen_w(7, 96, seed=4))
    y1 = orc.gemm(_bits(x), w)
    x8 = (x.float() * 8.0).to(torch.bfloat16)           # exact: exponent + 3
    y8 = orc.gemm(_bits(x8), w)
    assert np.array_equal(y8, 8.0 * y1)
    w_half = _bits((torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).float() * 0.5)
                   .to(torch.bfloat16))
    y_half = orc.gemm(_bits(x), w_half)
    assert np.array_equal(y_half, 0.5 * y1)


def pin_row_independence(orc):
    x = _bits(gen_x(5, 160, seed=5))
    w = _bits(gen_w(9, 160, seed=6))
    y = orc.gemm(x, w)
    for m in range(5):
        ym = orc.gemm(x[m:m + 1], w)
        assert np.array_equal(ym[0], y[m])


def pin_thread_invariance(orc):
    x = _bits(gen_x(3, 256, seed=7))
    w = _bits(gen_w(37, 256, seed=8))
    assert np.array_equal(orc.gemm(x, w, nthreads=1), orc.gemm(x, w, nthreads=5))


def pin_brute_force_exact(orc):
    # bf16 values are dyadic rationals: the exact sum is a Fraction, and the
    # double oracle (exact products, K-1 rounded additions) must sit within
    # gamma_K * sum|x*w| of it, gamma_K = K*u/(1-K*u), u = 2^-53.
    u = Fraction(1, 1 << 53)
    for (M, N, K, seed) in ((1, 1, 1, 0), (2, 3, 7, 1), (3, 5, 33, 2), (2, 4, 64, 3), (1, 2, 200, 4)):
        x = _bits(gen_x(M, K, seed=100 + seed, dist="uniform"))
        w = _bits(gen_w(N, K, seed=200 + seed, std=1.0))
        y = orc.gemm(x, w)
        for m in range(M):
            for n in range(N):
                terms = [bf16_exact(int(x[m, k])) * bf16_exact(int(w[n, k])) for k in range(K)]
                exact = sum(terms, Fraction(0))
                mag = sum((abs(t) for t in terms), Fraction(0))
                gamma = K * u / (1 - K * u)
                err = abs(Fraction(float(y[m, n])) - exact)
                assert err <= gamma * mag, f"({M},{N},{K}) y[{m},{n}] off by {float(err)}"


def pin_kda_chain_closed_form(orc):
    # x = 1, Q/K/V/G rows = 2^-10, F_A/beta rows = 1 + 2^-7, W_fb = 1, K = 7168:
    #   qkvg = 7168 * 2^-10 = 7 exactly
    #   fab  = 7168 * (1 + 2^-7) = 7224 exactly (in double)
    #   f_a  = bf16(7224) = 7232 (ulp 32 at 2^12, 7224/32 = 225.75 -> 226)
    #   fb   = 128 * 7232 = 925696
    M, K, Nq, Nfab, Nfb = 2, 7168, 32, 136, 16
    x = _const_bf16((M, K), 1.0)
    wp = np.concatenate([_const_bf16((Nq, K), 2.0 ** -10), _const_bf16((Nfab, K), 1.0 + 2.0 ** -7)])
    wfb = _const_bf16((Nfb, 128), 1.0)
    qkvg, fab, fa, fb = orc.kda_proj(x, wp, wfb, Nq, Nfab)
    assert np.array_equal(qkvg, np.full((M, Nq), 7.0))
    assert np.array_equal(fab, np.full((M, Nfab), 7224.0))
    assert np.array_equal(fa, np.full((M, 128), 0x45E2, dtype=np.uint16))
    assert np.array_equal(fb, np.full((M, Nfb), 925696.0))


def pin_kda_slices(orc):
    # the packed projection equals separate GEMMs over the row slices; F_B
    # consumes the bf16 F_A half (columns 0..127 of the F_A/beta output)
    M, K, Nq, Nfab, Nfb = 3, 256, 40, 136, 24
    x = _bits(gen_x(M, K, seed=9))
    wp = _bits(gen_w(Nq + Nfab, K, seed=10))
    wfb = _bits(gen_w(Nfb, 128, seed=12, std=0.5))
    qkvg, fab, fa, fb = orc.kda_proj(x, wp, wfb, Nq, Nfab)
    assert np.array_equal(qkvg, orc.gemm(x, wp[:Nq]))
    assert np.array_equal(fab, orc.gemm(x, wp[Nq:]))
    for m in range(M):
        for j in (0, 1, 64, 127):
            # nearest bf16 to the double F_A value, by exact comparison
            v = Fraction(float(fab[m, j]))
            got = bf16_exact(int(fa[m, j]))
            assert abs(got - v) <= abs(v) * Fraction(1, 256), "F_A not the rounded F_A/beta column"
    assert np.array_equal(fb, orc.gemm(fa, wfb))


def pin_fp16_golden(orc):
    cases = load_fp16_cases()
    bits = np.array([c[0] for c in cases], dtype=np.uint16)
    got = orc.fp16_to_f64(bits)
    for (b, want, line), g in zip(cases, got.tolist()):
        if np.isnan(want):
            assert np.isnan(g), f"fp16 {b:04X} -> {g!r}, want NaN  [{line}]"
        else:
            assert g == want and np.signbit(g) == np.signbit(want), \
                f"fp16 {b:04X} -> {g!r}, want {want!r}  [{line}]"


def pin_fp16_widen_exact(orc):
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 10) & 0x1F) != 0x1F]
    got = orc.fp16_to_f64(bits)
    for b, g in zip(bits.tolist(), got.tolist()):
        assert Fraction(g) == fp16_exact(b), f"widen fp16 {b:04X} = {g!r}"


def pin_gemm_ex_closed_forms(orc):
    # all ones: K exactly; plus a residual r: K + r exactly (one addition)
    for dtype in ("bf16", "fp16"):
        for K in (1, 64, 1024, 7168):
            x = _const((2, K), 1.0, dtype)
            w = _const((3, K), 1.0, dtype)
            assert np.array_equal(orc.gemm_ex(x, w, None, dtype), np.full((2, 3), float(K)))
            r = np.stack([_const((3,), v, dtype) for v in (0.5, -3.0)])
            y = orc.gemm_ex(x, w, r, dtype)
            assert np.array_equal(y, np.array([[K + 0.5] * 3, [K - 3.0] * 3])), f"{dtype} K={K}: {y}"
        # x = 0: the residual itself, element by element
        M, N, K = 3, 5, 40
        res = bits16(gen_x(M, N, seed=21, dtype=torch.float16 if dtype == "fp16" else torch.bfloat16))
        y = orc.gemm_ex(_const((M, K), 0.0, dtype), _const((N, K), 1.0, dtype), res, dtype)
        for m in range(M):
            for n in range(N):
                assert Fraction(float(y[m, n])) == _exact(int(res[m, n]), dtype), f"{dtype} y[{m},{n}]"


def pin_fp16_one_hot(orc):
    M, K, N = 3, 48, 10
    w = bits16(gen_w(N, K, seed=13, std=1.0, dtype=torch.float16))
    cols = [0, 47, 9]
    xf = torch.zeros(M, K)
    for m, j in enumerate(cols):
        xf[m, j] = 1.0
    y = orc.gemm_ex(bits16(xf.to(torch.float16)), w, None, "fp16")
    for m, j in enumerate(cols):
        for n in range(N):
            assert Fraction(float(y[m, n])) == fp16_exact(int(w[n, j])), f"y[{m},{n}] != W[{n},{j}]"


def pin_gemm_ex_brute_force(orc):
    # exact rational sum + residual; the double result sits within
    # gamma_{K+1} * (sum|x*w| + |r|) of it
    u = Fraction(1, 1 << 53)
    for dtype, tdt in (("bf16", torch.bfloat16), ("fp16", torch.float16)):
        for (M, N, K, seed) in ((1, 2, 5, 0), (2, 3, 31, 1), (3, 2, 70, 2)):
            x = bits16(gen_x(M, K, seed=300 + seed, dist="uniform", dtype=tdt))
            w = bits16(gen_w(N, K, seed=400 + seed, std=1.0, dtype=tdt))
            r = bits16(gen_x(M, N, seed=500 + seed, dtype=tdt))
            y = orc.gemm_ex(x, w, r, dtype)
            for m in range(M):
                for n in range(N):
                    terms = [_exact(int(x[m, k]), dtype) * _exact(int(w[n, k]), dtype) for k in range(K)]
                    rv = _exact(int(r[m, n]), dtype)
                    exact = sum(terms, Fraction(0)) + rv
                    mag = sum((abs(t) for t in terms), Fraction(0)) + abs(rv)
                    gamma = (K + 1) * u / (1 - (K + 1) * u)
                    err = abs(Fraction(float(y[m, n])) - exact)
                    assert err <= gamma * mag, f"{dtype} ({M},{N},{K}) y[{m},{n}] off by {float(err)}"


PINS = [
    pin_rne_golden,
    pin_fp16_golden,
    pin_fp16_widen_exact,
    pin_gemm_ex_closed_forms,
    pin_fp16_one_hot,
    pin_gemm_ex_brute_force,
    pin_widen_exact,
    pin_all_ones,
    pin_one_hot,
    pin_pow2_scaling,
    pin_row_independence,
    pin_thread_invariance,
    pin_brute_force_exact,
    pin_kda_chain_closed_form,
    pin_kda_slices,
]
