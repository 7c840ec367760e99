"""skinny_gemm_ex on the GPU vs the CPU oracle: fp16 inputs and the residual add
of the skinny GEMM (Kimi K3 support page, part 1, CuteSkinnyGemm: C = A * B^T
+ residual, bf16/fp16 inputs, fp32 accumulation).

Tolerance: |gpu - ref| <= 4 ulp(|ref|) + 1e-3 per element, ulp of the output
type (bf16: 8 significant bits, fp16: 11); outputs are NaN-poisoned first.
Every kernel kind runs with both element types, with and without a residual,
on ragged shapes; closed forms pin the residual's place in the sum exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg
from decode_projection_gemms_gb300.inputs import bits16, gen_w, gen_x

from gpu_helpers import NTHREADS, to_f64

pytestmark = pytest.mark.gpu

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    yield
    assert binding.device_error() == 0


def case(M, N, K, dtype, seed, residual=True):
    tdt = DTYPES[dtype]
    x = gen_x(M, K, seed=seed, dtype=tdt)
    W = gen_w(N, K, seed=seed + 1, dtype=tdt)
    r = gen_x(M, N, seed=seed + 2, dtype=tdt) if residual else None
    return x, W, r


def check_ex(x, W, r, dtype, cfg, label=""):
    M, N = x.shape[0], W.shape[0]
    y = torch.full((M, N), float("nan"), dtype=DTYPES[dtype], device="cuda")
    binding.skinny_gemm_ex(x.cuda(), W.cuda(), r.cuda() if r is not None else None, y, cfg=cfg)
    torch.cuda.synchronize()
    ref = oracle.gemm_ex(bits16(x), bits16(W), bits16(r) if r is not None else None, dtype,
                         nthreads=NTHREADS)
    res = oracle.compare(to_f64(y), ref, dtype=dtype)
    assert res["ok"], f"{label} {dtype} M={M} N={N} K={x.shape[1]} cfg={cfg.as_dict() if cfg else 'auto'}: {res}"
    return y


CONFIGS = {
    "cc_split4": KpCfg.make("cc", split_k=4, block=256, rows=2, k_unroll=2),
    "cc_split1": KpCfg.make("cc", split_k=1, block=128, rows=1, k_unroll=4),
    # the shared-memory ring form, one K slice and three
    "cc_ring_split1": KpCfg.make("cc", split_k=1, block=256, rows=2, k_unroll=2, stages=4),
    "cc_ring_split3": KpCfg.make("cc", split_k=3, block=128, rows=4, k_unroll=1, stages=4),
    "tc05_c1": KpCfg.make("tc05", split_k=1, k_unroll=2),
    "tc05_c4": KpCfg.make("tc05", split_k=4, k_unroll=2, stages=3),
    "tc05_c16": KpCfg.make("tc05", split_k=16, k_unroll=1),
    "auto": None,
}


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("name", sorted(CONFIGS))
@pytest.mark.parametrize("M", [1, 5, 16])
def test_ex_kernels(dtype, residual, name, M):
    cfg = CONFIGS[name]
    if cfg is not None:
        try:
            binding.scratch_bytes(M, 1000, 7168, cfg, 152)
        except binding.KdaProjError as e:
            assert e.code == binding.KP_ECONFIG
            pytest.skip("configuration not valid at this M (x slice too large)")
    x, W, r = case(M, 1000, 7168, dtype, seed=40 + M, residual=residual)
    check_ex(x, W, r, dtype, cfg, name)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M", [17, 64, 129, 256, 300])
def test_ex_tc05_large_m(dtype, M):
    # ragged N and a partial last K block; M = 300 runs as two token tiles
    x, W, r = case(M, 264, 1032, dtype, seed=M)
    for C in (1, 4):
        check_ex(x, W, r, dtype, KpCfg.make("tc05", split_k=C, k_unroll=1), f"tc05 C={C}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M", [3, 128])
def test_ex_tc05_odd_n(dtype, M):
    # the general epilogue's split-K reduction with N not a multiple of 4
    x, W, r = case(M, 1001, 2048, dtype, seed=M + 5)
    for C in (2, 8):
        check_ex(x, W, r, dtype, KpCfg.make("tc05", split_k=C, k_unroll=1, stages=2), f"tc05 C={C}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("M", [1, 33])
def test_ex_smallk(dtype, M):
    x, W, r = case(M, 1024, 128, dtype, seed=70 + M)
    check_ex(x, W, r, dtype, KpCfg.make("smallk", block=256, rows=8), "smallk")
    check_ex(x, W, None, dtype, KpCfg.make("smallk", block=128, rows=16), "smallk")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_ex_residual_in_place(dtype, name):
    # residual is y itself: each element is read before it is written
    M = 4
    x, W, r = case(M, 520, 2048, dtype, seed=90)
    ref = oracle.gemm_ex(bits16(x), bits16(W), bits16(r), dtype, nthreads=NTHREADS)
    y = r.cuda().clone()
    binding.skinny_gemm_ex(x.cuda(), W.cuda(), y, y, cfg=CONFIGS[name])
    torch.cuda.synchronize()
    res = oracle.compare(to_f64(y), ref, dtype=dtype)
    assert res["ok"], f"{name} in place: {res}"


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_ex_closed_forms(name):
    cfg = CONFIGS[name]
    # all ones: K + r exactly (fp16: 1024 - 24 = 1000; bf16: 7168 + 64 = 7232)
    for dtype, K, rv in (("fp16", 1024, -24.0), ("bf16", 7168, 64.0)):
        tdt = DTYPES[dtype]
        M, N = 3, 300
        x = torch.ones((M, K), dtype=tdt, device="cuda")
        W = torch.ones((N, K), dtype=tdt, device="cuda")
        r = torch.full((M, N), rv, dtype=tdt, device="cuda")
        y = binding.skinny_gemm_ex(x, W, r, cfg=cfg)
        torch.cuda.synchronize()
        assert torch.equal(y.float().cpu(), torch.full((M, N), K + rv)), f"{name} {dtype}"
        # x = 0: exactly the residual
        r = gen_x(M, N, seed=5, dtype=tdt).cuda()
        y = binding.skinny_gemm_ex(torch.zeros_like(x), W, r, cfg=cfg)
        torch.cuda.synchronize()
        assert torch.equal(y, r), f"{name} {dtype}: x = 0 must give the residual"


@pytest.mark.parametrize("name", ["cc_split4", "tc05_c4", "auto"])
def test_ex_fp16_one_hot(name):
    # a one-hot row of x selects a column of W exactly, in fp16
    M, K, N = 3, 2048, 136
    W = gen_w(N, K, seed=3, std=1.0, dtype=torch.float16)
    cols = [0, 2047, 777]
    x = torch.zeros((M, K), dtype=torch.float16)
    for m, j in enumerate(cols):
        x[m, j] = 1.0
    y = binding.skinny_gemm_ex(x.cuda(), W.cuda(), cfg=CONFIGS[name])
    torch.cuda.synchronize()
    for m, j in enumerate(cols):
        assert torch.equal(y[m].cpu(), W[:, j]), f"{name} row {m}"


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_ex_bf16_without_residual_is_skinny_gemm(name):
    x, W, _ = case(8, 700, 4096, "bf16", seed=11, residual=False)
    x, W = x.cuda(), W.cuda()
    a = binding.skinny_gemm(x, W, cfg=CONFIGS[name])
    b = binding.skinny_gemm_ex(x, W, cfg=CONFIGS[name])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_ex_rejects_mixed_types():
    x = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    W = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        binding.skinny_gemm_ex(x, W)
