"""Token counts above 256 (prefill) in one tcgen05 launch: token tiles of 256
along the grid's second axis, against the CPU oracle.

Where a full oracle product would be slow, a seeded sample of output columns
is compared (each output is an independent dot product). Full 256-token tiles
run exactly the per-tile MMA sequence of a separate 256-token call, so those
rows must be bit-identical to per-tile calls with the same configuration.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg
from decode_projection_gemms_gb300.inputs import bf16_bits, bits16, gen_w, gen_x

from gpu_helpers import NTHREADS, poisoned, to_f64

pytestmark = pytest.mark.gpu

MAX_ORACLE_MACS = 1 << 27


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    yield
    assert binding.device_error() == 0


def sampled_check(y, x_bits, w_bits, label, dtype="bf16", res_bits=None, seed=0):
    M, N = y.shape
    K = x_bits.shape[1]
    got = to_f64(y)
    assert np.isfinite(got).all(), f"{label}: unwritten outputs"
    ncols = N if M * N * K <= MAX_ORACLE_MACS else max(8, MAX_ORACLE_MACS // (M * K))
    rng = np.random.default_rng(seed)
    cols = np.arange(N) if ncols >= N else np.sort(rng.choice(N, size=ncols, replace=False))
    cols = np.unique(np.concatenate([cols, [0, N - 1]]))
    r = res_bits[:, cols] if res_bits is not None else None
    ref = oracle.gemm_ex(x_bits, w_bits[cols], r, dtype, nthreads=NTHREADS)
    c = oracle.compare(got[:, cols], ref, dtype=dtype)
    assert c["ok"], f"{label} ({len(cols)} columns): {c}"


CONFIGS = [None, KpCfg.make("tc05", split_k=1, k_unroll=1), KpCfg.make("tc05", split_k=4, k_unroll=2, stages=2),
           # 256-row CTAs with cluster split-K (the table's M = 512 and 1024 prefill entries)
           KpCfg.make("tc05", split_k=4, rows=256, k_unroll=1),
           KpCfg.make("tc05", split_k=2, rows=256, k_unroll=1, stages=3)]


@pytest.mark.parametrize("M", [257, 300, 513, 1024])
@pytest.mark.parametrize("N,K", [(264, 1032), (1000, 7168)])
@pytest.mark.parametrize("ci", range(len(CONFIGS)))
def test_prefill_parity(M, N, K, ci):
    x = gen_x(M, K, seed=M + 3)
    W = gen_w(N, K, seed=N + 5)
    y = poisoned((M, N))
    binding.skinny_gemm(x.cuda(), W.cuda(), y, cfg=CONFIGS[ci])
    torch.cuda.synchronize()
    sampled_check(y, bf16_bits(x), bf16_bits(W), f"M={M} N={N} K={K} cfg#{ci}", seed=M)


@pytest.mark.parametrize("cfg", [KpCfg.make("tc05", split_k=1, k_unroll=1),
                                 KpCfg.make("tc05", split_k=8, k_unroll=2, stages=2)])
def test_prefill_full_tiles_match_per_tile_calls(cfg):
    M, N, K = 768, 520, 2048
    x = gen_x(M, K, seed=1).cuda()
    W = gen_w(N, K, seed=2).cuda()
    y = binding.skinny_gemm(x, W, cfg=cfg)
    parts = [binding.skinny_gemm(x[m:m + 256].contiguous(), W, cfg=cfg) for m in range(0, M, 256)]
    torch.cuda.synchronize()
    assert torch.equal(y, torch.cat(parts))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_prefill_residual(dtype):
    # the general kernel: residual rows offset by each token tile's first token
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    M, N, K = 600, 392, 1024
    x = gen_x(M, K, seed=7, dtype=tdt)
    W = gen_w(N, K, seed=8, dtype=tdt)
    r = gen_x(M, N, seed=9, dtype=tdt)
    for cfg in (KpCfg.make("tc05", split_k=1, k_unroll=1), KpCfg.make("tc05", split_k=2, k_unroll=2)):
        y = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        binding.skinny_gemm_ex(x.cuda(), W.cuda(), r.cuda(), y, cfg=cfg)
        torch.cuda.synchronize()
        sampled_check(y, bits16(x), bits16(W), f"{dtype} residual", dtype=dtype, res_bits=bits16(r))


def test_prefill_default_large_grid():
    # more 128-row CTAs than SMs: the built-in rule switches to 256-row CTAs
    M, N, K = 2560, 4096, 1024
    cfg = binding.select_config(M, N, K, 152)
    x = gen_x(M, K, seed=21)
    W = gen_w(N, K, seed=22)
    y = poisoned((M, N))
    binding.skinny_gemm(x.cuda(), W.cuda(), y)
    torch.cuda.synchronize()
    sampled_check(y, bf16_bits(x), bf16_bits(W), f"default {cfg.as_dict()}", seed=3)


def test_prefill_closed_form():
    # all ones over 2048 tokens in 8 token tiles: every output is K exactly
    M, N, K = 2048, 136, 7168
    x = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
    y = binding.skinny_gemm(x, W)
    torch.cuda.synchronize()
    assert torch.equal(y.float().cpu(), torch.full((M, N), float(K)))
