"""The shape-dynamic skinny GEMM over the sweep grid (M up to 256 x N in {136,
512, 1024, 4096, 8192} x K in {128, 1024, 7168, 16384}) with the configuration
the table (or the built-in rule) picks, against the CPU oracle.

Where the oracle would take too long for every output (large M * N * K), a
seeded sample of output columns is compared: each output is an independent dot
product, so a column the oracle computes alone is exactly that column of the
full product. Tolerance as everywhere: 4 ulp_bf16 + 1e-3, NaN-poisoned outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.inputs import bf16_bits, gen_w, gen_x

from gpu_helpers import NTHREADS, poisoned, to_f64

pytestmark = pytest.mark.gpu

SWEEP_N = [136, 512, 1024, 4096, 8192]
SWEEP_K = [128, 1024, 7168, 16384]
MS = [1, 7, 16, 24, 129, 256]
MAX_ORACLE_MACS = 1 << 27   # per case; beyond it, sampled columns


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    yield
    assert binding.device_error() == 0


@pytest.mark.parametrize("K", SWEEP_K)
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep_grid_auto_config(N, K):
    W = gen_w(N, K, seed=N + K)
    Wd = W.cuda()
    wb = bf16_bits(W)
    rng = np.random.default_rng(N * 7 + K)
    for M in MS:
        x = gen_x(M, K, seed=M + N + K)
        y = poisoned((M, N))
        binding.skinny_gemm(x.cuda(), Wd, y)          # table / built-in choice
        torch.cuda.synchronize()
        got = to_f64(y)
        assert np.isfinite(got).all(), f"M={M} N={N} K={K}: unwritten outputs"
        ncols = N if M * N * K <= MAX_ORACLE_MACS else max(8, MAX_ORACLE_MACS // (M * K))
        cols = np.arange(N) if ncols >= N else np.sort(rng.choice(N, size=ncols, replace=False))
        # always include both ends (first and ragged last tile)
        cols = np.unique(np.concatenate([cols, [0, N - 1]]))
        ref = oracle.gemm(bf16_bits(x), wb[cols], nthreads=NTHREADS)
        r = oracle.compare(got[:, cols], ref)
        cfg = binding.select_config(M, N, K, 152).as_dict()
        assert r["ok"], f"M={M} N={N} K={K} cfg={cfg} ({len(cols)} columns): {r}"


def test_sweep_every_small_m():
    # M = 1..16 one by one (the CUDA-core kernel's unrolled token counts)
    N, K = 512, 1024
    W = gen_w(N, K, seed=5)
    for M in range(1, 17):
        x = gen_x(M, K, seed=M)
        y = poisoned((M, N))
        binding.skinny_gemm(x.cuda(), W.cuda(), y)
        torch.cuda.synchronize()
        r = oracle.compare(to_f64(y), oracle.gemm(bf16_bits(x), bf16_bits(W), nthreads=NTHREADS))
        assert r["ok"], f"M={M}: {r}"
