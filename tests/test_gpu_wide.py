"""The tcgen05 kernel with 256 feature rows per CTA (configuration rows = 256):
two 128-row MMAs on the same x operand into two TMEM accumulators. Parity
against the CPU oracle on ragged shapes and every cluster size, the cluster
reduction over 256 rows, the fused F_B and the single launch over the packed
weight, prefill token tiles, fp16 and the residual.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg
from decode_projection_gemms_gb300.inputs import bf16_bits, bits16, gen_w, gen_x

from gpu_helpers import NTHREADS, check_gemm, check_kda, gemm_case, kda_inputs, poisoned, to_f64

pytestmark = pytest.mark.gpu


def wide(C, nkb=2, stages=0, flags=binding.FLAG_PDL, producers=1):
    return KpCfg.make("tc05", split_k=C, rows=256, k_unroll=nkb, stages=stages, flags=flags,
                      producers=producers)


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    yield
    assert binding.device_error() == 0


def valid(M, N, K, cfg):
    try:
        binding.scratch_bytes(M, N, K, cfg, 152)
        return True
    except binding.KdaProjError as e:
        assert e.code == binding.KP_ECONFIG
        return False


@pytest.mark.parametrize("M", [1, 16, 64, 128, 200, 256])
@pytest.mark.parametrize("N,K", [(136, 7168), (1000, 1032), (4096, 2048)])
@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_wide_shapes(M, N, K, C):
    cfg = wide(C, nkb=1 if M > 128 else 2)
    if not valid(M, N, K, cfg):
        pytest.skip("does not fit")
    x, W = gemm_case(M, N, K, seed=M + N + C)
    check_gemm(x, W, cfg, f"wide C={C}")


@pytest.mark.parametrize("C", [1, 4, 8])
def test_wide_matches_narrow_rows(C):
    # same K split, each row's MMA chain unchanged: 256-row CTAs give the
    # 128-row CTAs' results bit for bit
    x, W = gemm_case(32, 1000, 7168, seed=4)
    x, W = x.cuda(), W.cuda()
    a = binding.skinny_gemm(x, W, cfg=KpCfg.make("tc05", split_k=C, k_unroll=2))
    b = binding.skinny_gemm(x, W, cfg=wide(C))
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("M", [300, 1024])
def test_wide_prefill(M):
    N, K = 520, 2048
    x, W = gemm_case(M, N, K, seed=M)
    for C in (1,):   # split-K would need a 256 x 256 fp32 partial tile: does not fit
        y = poisoned((M, N))
        binding.skinny_gemm(x.cuda(), W.cuda(), y, cfg=wide(C, nkb=1))
        torch.cuda.synchronize()
        cols = np.unique(np.concatenate([np.arange(0, N, 7), [N - 1]]))
        ref = oracle.gemm(bf16_bits(x), bf16_bits(W)[cols], nthreads=NTHREADS)
        r = oracle.compare(to_f64(y)[:, cols], ref)
        assert r["ok"], f"wide prefill M={M} C={C}: {r}"


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_wide_residual(dtype):
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    M, N, K = 40, 600, 3072
    x = gen_x(M, K, seed=1, dtype=tdt)
    W = gen_w(N, K, seed=2, dtype=tdt)
    r = gen_x(M, N, seed=3, dtype=tdt)
    for C in (1, 4):
        y = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        binding.skinny_gemm_ex(x.cuda(), W.cuda(), r.cuda(), y, cfg=wide(C))
        torch.cuda.synchronize()
        ref = oracle.gemm_ex(bits16(x), bits16(W), bits16(r), dtype, nthreads=NTHREADS)
        c = oracle.compare(to_f64(y), ref, dtype=dtype)
        assert c["ok"], f"{dtype} C={C}: {c}"


# ---- the projection with 256-row CTAs ----------------------------------------------------

@pytest.fixture(scope="module")
def plan():
    p = binding.KdaPlan(K=7168, N_qkvg=4096, N_fab=136, N_fb=1024, max_M=256)
    yield p
    p.close()


def _run_mode(plan, x, wp, wfb, mode, aux, evs):
    M = x.shape[0]
    outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
    plan.set_overlap(mode)
    plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
    torch.cuda.synchronize()
    return [o.clone() for o in outs]


@pytest.mark.parametrize("M", [1, 16, 64, 128])
@pytest.mark.parametrize("C", [2, 4, 8, 16])
def test_wide_single_launch_and_fused(plan, M, C):
    cq = wide(C, nkb=2 if M <= 64 else 1)
    cf = wide(C, nkb=2 if M <= 64 else 1, flags=binding.FLAG_PDL | binding.FLAG_FUSE_FB)
    saved = [plan.get_config(b, M) for b in range(3)]
    try:
        try:
            plan.set_config(binding.BRANCH_QKVG, M, cq)
            plan.set_config(binding.BRANCH_FAB, M, cf)
        except binding.KdaProjError as e:
            pytest.skip(str(e))
        x, wp, wfb = kda_inputs(M, layer=9, seed=12)
        x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
        aux = torch.cuda.Stream()
        evs = binding.make_events()
        one = _run_mode(plan, x, wp, wfb, 2, aux, evs)
        check_kda(one, x.cpu(), wp.cpu(), wfb.cpu(), 4096, 136, f"wide single launch C={C} M={M}")
        ovl = _run_mode(plan, x, wp, wfb, 1, aux, evs)
        check_kda(ovl, x.cpu(), wp.cpu(), wfb.cpu(), 4096, 136, f"wide fused aux C={C} M={M}")
        # same configuration and K split for both: identical outputs
        for a, b in zip(one, ovl):
            assert torch.equal(a, b)
        ref_fb = binding.skinny_gemm(one[1][:, :128].contiguous(), wfb,
                                     cfg=KpCfg.make("tc05", split_k=1, k_unroll=2))
        torch.cuda.synchronize()
        assert torch.equal(ref_fb, one[2])
    finally:
        for b, c in enumerate(saved):
            plan.set_config(b, M, c)
        plan.set_overlap(-1)
