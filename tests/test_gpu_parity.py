"""CUDA path vs the CPU oracle, element by element, on the same seeded inputs.

Tolerance (bf16 output, fp32 accumulation): |gpu - ref| <= 4 ulp_bf16(|ref|)
+ 1e-3 per element; outputs are NaN-poisoned before each call so an element a
kernel never writes fails. F_B is checked twice: from the GPU's own bf16 F_A
at that plain bound (stage-isolated), and end to end from the oracle's F_A,
where the bound adds the propagated F_A tolerance (sum_k dF_A[k] |W_fb[n, k]|).
"""
import numpy as np
import pytest
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg
from decode_projection_gemms_gb300.inputs import bf16_bits, gen_w, gen_x

from gpu_helpers import (NTHREADS, check_gemm, check_kda, gemm_case, kda_inputs,
                         kda_reference, poisoned, to_f64)

pytestmark = pytest.mark.gpu

CC_VARIANTS = [(1, 4), (2, 2), (2, 4), (4, 1), (4, 2), (8, 1)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    yield
    assert binding.device_error() == 0


# ---- single skinny GEMM: M=1, K=2048, N=1024, x ~ U(-1, 1), seed 0 -------------------

def config1():
    return gemm_case(1, 1024, 2048, seed=0, dist="uniform")


def test_config1_auto():
    x, W = config1()
    check_gemm(x, W, None, "auto")


@pytest.mark.parametrize("R,U", CC_VARIANTS)
@pytest.mark.parametrize("S", [1, 3, 8])
def test_config1_cc(R, U, S):
    x, W = config1()
    check_gemm(x, W, KpCfg.make("cc", split_k=S, block=256, rows=R, k_unroll=U), "cc")


@pytest.mark.parametrize("C,nkb,stages", [(1, 1, 0), (2, 4, 2), (4, 2, 3), (16, 4, 0), (8, 1, 5),
                                           (32, 1, 0)])
def test_config1_tc05(C, nkb, stages):
    x, W = config1()
    cfg = KpCfg.make("tc05", split_k=C, k_unroll=nkb, stages=stages)
    if C == 32:  # clusters hold at most 16 CTAs
        with pytest.raises(binding.KdaProjError) as e:
            binding.skinny_gemm(x.cuda(), W.cuda(), cfg=cfg)
        assert e.value.code == binding.KP_ECONFIG
        return
    check_gemm(x, W, cfg, "tc05")


# ---- CUDA-core kernel: every M bucket, ragged N, several K -------------------------------

@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 11, 16])
@pytest.mark.parametrize("N,K", [(136, 7168), (1000, 1024), (4096, 1032)])
def test_cc_shapes(M, N, K):
    x, W = gemm_case(M, N, K, seed=M)
    for R, U in CC_VARIANTS:
        cfg = KpCfg.make("cc", split_k=5, block=256, rows=R, k_unroll=U)
        try:
            binding.scratch_bytes(M, N, K, cfg, 152)
        except binding.KdaProjError:
            continue  # variant not built for this M
        check_gemm(x, W, cfg, "cc")


def test_cc_block_sizes_and_unsplit():
    x, W = gemm_case(3, 777, 2048, seed=5)
    for block in (32, 128, 256, 512):
        for S in (1, 2, 16):
            check_gemm(x, W, KpCfg.make("cc", split_k=S, block=block, rows=2, k_unroll=2), "cc")


# ---- CUDA-core kernel, shared-memory ring form (stages = 4) --------------------------------

def _cc_ok(M, N, K, cfg):
    try:
        binding.scratch_bytes(M, N, K, cfg, 152)
        return True
    except binding.KdaProjError:
        return False


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 11, 16])
@pytest.mark.parametrize("N,K", [(136, 7168), (1000, 1024), (4096, 1032), (77, 40)])
def test_cc_ring_shapes(M, N, K):
    """The ring form against the oracle, and bit for bit against the register
    form of the same configuration: both take each lane's chunks in the same
    order, so the sums are the same."""
    x, W = gemm_case(M, N, K, seed=M + 40)
    ran = 0
    for R, U in CC_VARIANTS:
        for S, block in ((1, 256), (5, 128), (3, 448)):
            ring = KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U, stages=4)
            if not _cc_ok(M, N, K, ring):
                continue
            y, _ = check_gemm(x, W, ring, "cc ring")
            plain = KpCfg.make("cc", split_k=S, block=block, rows=R, k_unroll=U)
            y0 = binding.skinny_gemm(x.cuda(), W.cuda(), cfg=plain)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), y0.view(torch.int16)), (M, N, K, R, U, S, block)
            ran += 1
    assert ran > 0


def test_cc_ring_full_size_qkvg():
    """The ring form at the Q/K/V/G shape (M = 4, N = 4096, K = 7168) with
    one K slice and 14 warps per CTA (the launch shape the benchmark times),
    on sampled outputs."""
    M, N, K = 4, 4096, 7168
    x, W = gemm_case(M, N, K, seed=3)
    cfg = KpCfg.make("cc", split_k=1, block=448, rows=2, k_unroll=2, stages=4)
    y = binding.skinny_gemm(x.cuda(), W.cuda(), cfg=cfg)
    torch.cuda.synchronize()
    cols = torch.arange(0, N, 37)
    ref = oracle.gemm(bf16_bits(x), bf16_bits(W[cols]), nthreads=NTHREADS)
    r = oracle.compare(to_f64(y[:, cols]), ref)
    assert r["ok"], r


def test_cc_ring_rejects_what_does_not_fit():
    """Only a 4-slot ring is built, and the x slice plus the ring must fit in
    shared memory."""
    assert not _cc_ok(4, 4096, 7168, KpCfg.make("cc", split_k=1, rows=2, k_unroll=2, stages=3))
    # x slice 8 x 7168 x 2 = 112 KB, ring 16 warps x 4 x 4 x 2 x 512 B = 256 KB
    assert not _cc_ok(8, 4096, 7168, KpCfg.make("cc", split_k=1, block=512, rows=4, k_unroll=2, stages=4))
    assert _cc_ok(8, 4096, 7168, KpCfg.make("cc", split_k=2, block=256, rows=2, k_unroll=2, stages=4))


# ---- tcgen05 kernel: token counts across the UMMA N range, ragged N and K -----------------

TC05_VARIANTS = [(1, 2, 1), (4, 1, 1), (16, 4, 4), (8, 2, 2), (4, 4, 3)]


def _tc05_ok(M, N, K, cfg):
    try:
        binding.scratch_bytes(M, N, K, cfg, 152)
        return True
    except binding.KdaProjError:
        return False


@pytest.mark.parametrize("M", [1, 8, 16, 17, 48, 64, 100, 128, 129, 256])
@pytest.mark.parametrize("N,K", [(136, 7168), (1000, 1032), (4096, 1024)])
def test_tc05_shapes(M, N, K):
    x, W = gemm_case(M, N, K, seed=100 + M)
    ran = 0
    for C, nkb, P in TC05_VARIANTS:
        cfg = KpCfg.make("tc05", split_k=C, k_unroll=nkb, producers=P)
        if _tc05_ok(M, N, K, cfg):
            check_gemm(x, W, cfg, "tc05")
            ran += 1
    assert ran >= 2


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("nkb", [1, 2, 4])
def test_tc05_cluster_splits(C, nkb):
    # K = 4288 -> 67 K blocks: uneven ranges per cluster rank and short last stages
    x, W = gemm_case(24, 520, 4096 + 64 * 3, seed=7)
    for P in sorted({1, 2, nkb, 5}):
        check_gemm(x, W, KpCfg.make("tc05", split_k=C, k_unroll=nkb, producers=P, stages=2),
                   f"tc05 P={P}")


@pytest.mark.parametrize("N", [7, 131, 1001])
@pytest.mark.parametrize("C", [2, 4, 8])
@pytest.mark.parametrize("M", [1, 37, 128])
def test_tc05_odd_n(M, C, N):
    # N not a multiple of 4: the split-K reduction stores element by element,
    # and the last tile ends inside a group of four rows
    x, W = gemm_case(M, N, 2048, seed=M + C + N)
    cfg = KpCfg.make("tc05", split_k=C, k_unroll=1, stages=2)
    if not _tc05_ok(M, N, 2048, cfg):
        pytest.skip("does not fit")
    check_gemm(x, W, cfg, "tc05 odd N")


def test_tc05_m_above_256_two_token_tiles():
    x, W = gemm_case(300, 264, 512, seed=8)
    check_gemm(x, W, KpCfg.make("tc05", split_k=4, k_unroll=1), "tc05")


def test_tiny_shapes():
    x, W = gemm_case(2, 1, 8, seed=9)
    check_gemm(x, W, KpCfg.make("tc05", split_k=1, k_unroll=1), "tc05 N=1 K=8")
    check_gemm(x, W, KpCfg.make("cc", split_k=1, block=32, rows=1, k_unroll=4), "cc N=1 K=8")
    check_gemm(x, W, KpCfg.make("smallk", block=64, rows=1), "smallk N=1 K=8")


# ---- small-K kernel (the F_B shape) --------------------------------------------------------

@pytest.mark.parametrize("M", [1, 7, 33, 128])
@pytest.mark.parametrize("N,K,rows", [(1024, 128, 16), (100, 256, 8), (1024, 128, 64)])
def test_smallk_shapes(M, N, K, rows):
    x, W = gemm_case(M, N, K, seed=200 + M)
    check_gemm(x, W, KpCfg.make("smallk", block=256, rows=rows), "smallk")


# ---- closed forms through the GPU path -----------------------------------------------------

@pytest.mark.parametrize("cfg", [KpCfg.make("cc", split_k=7, rows=4, k_unroll=2),
                                 KpCfg.make("tc05", split_k=4, k_unroll=4), None])
def test_all_ones_gives_k_exactly(cfg):
    M, N, K = 4, 300, 7168
    x = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
    y = poisoned((M, N))
    binding.skinny_gemm(x, W, y, cfg=cfg)
    torch.cuda.synchronize()
    assert torch.equal(y.float().cpu(), torch.full((M, N), 7168.0))


def test_one_hot_selects_a_weight_column():
    M, N, K = 5, 640, 2048
    W = gen_w(N, K, seed=3, std=1.0)
    cols = [0, 17, 1000, 2047, 64]
    x = torch.zeros((M, K))
    for m, j in enumerate(cols):
        x[m, j] = 1.0
    x = x.to(torch.bfloat16)
    for cfg in (KpCfg.make("cc", split_k=4, rows=2, k_unroll=2),
                KpCfg.make("tc05", split_k=8, k_unroll=2)):
        y = poisoned((M, N))
        binding.skinny_gemm(x.cuda(), W.cuda(), y, cfg=cfg)
        torch.cuda.synchronize()
        for m, j in enumerate(cols):
            assert torch.equal(y[m].cpu(), W[:, j])


# ---- the full KDA projection at the pages' per-rank shapes --------------------------------

@pytest.fixture(scope="module")
def plan():
    p = binding.KdaPlan(K=7168, N_qkvg=4096, N_fab=136, N_fb=1024, max_M=256)
    yield p
    p.close()


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64, 128])
def test_kda_full_size_overlapped(plan, M):
    x, wp, wfb = kda_inputs(M, layer=0)
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
    plan.set_overlap(1)
    try:
        plan.run(x.cuda(), wp.cuda(), wfb.cuda(), *outs, aux_stream=aux, events=evs)
        torch.cuda.synchronize()
    finally:
        plan.set_overlap(-1)
    check_kda(outs, x, wp, wfb, 4096, 136, f"M={M}")


@pytest.mark.parametrize("M", [3, 13, 129, 256])
def test_kda_other_token_counts(plan, M):
    x, wp, wfb = kda_inputs(M, layer=5, seed=2)
    outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
    plan.run(x.cuda(), wp.cuda(), wfb.cuda(), *outs)
    torch.cuda.synchronize()
    check_kda(outs, x, wp, wfb, 4096, 136, f"M={M}")


def test_kda_last_layer_of_the_stack(plan):
    # the benchmark rotates through 48 layers; layer 47 has its own seed
    x, wp, wfb = kda_inputs(16, layer=47)
    outs = plan.run(x.cuda(), wp.cuda(), wfb.cuda())
    torch.cuda.synchronize()
    check_kda(outs, x, wp, wfb, 4096, 136, "layer 47")


def test_kda_small_packed_shapes():
    # ragged Q/K/V/G width, F_A/beta width 136, non-multiple-of-64 K
    p = binding.KdaPlan(K=1032, N_qkvg=1000, N_fab=136, N_fb=200, max_M=40)
    try:
        for M in (1, 9, 40):
            x, wp, wfb = kda_inputs(M, layer=1, seed=4, K=1032, Nq=1000, Nfab=136, Nfb=200)
            outs = (poisoned((M, 1000)), poisoned((M, 136)), poisoned((M, 200)))
            p.run(x.cuda(), wp.cuda(), wfb.cuda(), *outs, aux_stream=torch.cuda.Stream(),
                  events=binding.make_events())
            torch.cuda.synchronize()
            check_kda(outs, x, wp, wfb, 1000, 136, f"small M={M}")
    finally:
        p.close()


def test_kda_chain_closed_form():
    # x = 1, Q/K/V/G rows 2^-10, F_A/beta rows 1 + 2^-7, W_fb = 1, K = 7168:
    # qkvg = 7, fab = 7224 -> bf16 7232, fb = 128 * 7232 = 925696 (the bf16 of
    # 925696 is 925696: 0x4962 = 1.765625 * 2^19)
    M = 3
    p = binding.KdaPlan(K=7168, N_qkvg=256, N_fab=136, N_fb=64, max_M=M)
    try:
        x = torch.ones((M, 7168), dtype=torch.bfloat16, device="cuda")
        wp = torch.cat([torch.full((256, 7168), 2.0 ** -10), torch.full((136, 7168), 1 + 2.0 ** -7)])
        wp = wp.to(torch.bfloat16).cuda()
        wfb = torch.ones((64, 128), dtype=torch.bfloat16, device="cuda")
        oq, of, ob = p.run(x, wp, wfb)
        torch.cuda.synchronize()
        assert torch.equal(oq.float().cpu(), torch.full((M, 256), 7.0))
        assert torch.equal(of.float().cpu(), torch.full((M, 136), 7232.0))
        assert torch.equal(ob.float().cpu(), torch.full((M, 64), 925696.0))
    finally:
        p.close()


# ---- F_B in every schedule, stage-isolated at the plain bound ---------------------------------

@pytest.mark.parametrize("layer", [0, 47])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64, 128])
def test_kda_every_mode_against_the_oracle(plan, M, layer):
    """Sequential, overlapped, single launch, and the aux branch with F_B fused
    into the F_A/beta launch: every output against the oracle, F_B also from
    the GPU's own F_A at 4 ulp + 1e-3 with no widening."""
    x, wp, wfb = kda_inputs(M, layer=layer)
    ref = kda_reference(x, wp, wfb, 4096, 136)
    xd, wpd, wfbd = x.cuda(), wp.cuda(), wfb.cuda()
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    saved = plan.get_config(binding.BRANCH_FAB, M)
    try:
        for mode in (0, 1, 2):
            outs = _run_mode(plan, xd, wpd, wfbd, mode, aux, evs)
            check_kda(outs, x, wp, wfb, 4096, 136, f"mode {mode} M={M} layer {layer}", ref=ref)
        fused = KpCfg.from_buffer_copy(saved)
        if fused.kind == binding.KIND_TC05:
            fused.flags |= binding.FLAG_FUSE_FB
            try:
                plan.set_config(binding.BRANCH_FAB, M, fused)
            except binding.KdaProjError:
                return   # no room for the F_B operands beside this configuration
            for mode in (0, 1):
                outs = _run_mode(plan, xd, wpd, wfbd, mode, aux, evs)
                check_kda(outs, x, wp, wfb, 4096, 136, f"fused F_B mode {mode} M={M}", ref=ref)
    finally:
        plan.set_config(binding.BRANCH_FAB, M, saved)
        plan.set_overlap(-1)


@pytest.mark.parametrize("M", [1, 5, 16, 17, 64, 128, 200, 256])
def test_tc05_f_b_shape_one_cta_per_tile(M):
    """The fused F_B's MMA sequence (one CTA per 128-row tile, K = 128 in two
    64-wide K blocks) as a plain GEMM on the F_B shape, against the oracle."""
    x, W = gemm_case(M, 1024, 128, seed=300 + M)
    check_gemm(x, W, KpCfg.make("tc05", split_k=1, k_unroll=2), "tc05 F_B shape")
    x, W = gemm_case(M, 1000, 128, seed=400 + M)
    check_gemm(x, W, KpCfg.make("tc05", split_k=1, k_unroll=2), "tc05 F_B shape, ragged N")


# ---- bit identity: sequential == overlapped == graph replay == PDL off ---------------------

def _run(plan, x, wp, wfb, overlap, aux, evs):
    M = x.shape[0]
    outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
    plan.set_overlap(1 if overlap else 0)
    plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
    torch.cuda.synchronize()
    return [o.clone() for o in outs]


@pytest.mark.parametrize("M", [1, 4, 14, 16, 64, 128])
def test_overlap_graph_pdl_bit_identical(plan, M):
    x, wp, wfb = kda_inputs(M, layer=2, seed=1)
    x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    try:
        seq = _run(plan, x, wp, wfb, False, aux, evs)
        ovl = _run(plan, x, wp, wfb, True, aux, evs)
        again = _run(plan, x, wp, wfb, True, aux, evs)
        for a, b, c in zip(seq, ovl, again):
            assert torch.equal(a, b) and torch.equal(a, c)

        # captured and replayed (overlapped: aux joins the capture via events[0])
        outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
        plan.set_overlap(1)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(seq, outs):
            assert torch.equal(a, b)

        # programmatic dependent launch off for every branch
        saved = [plan.get_config(b, M) for b in range(3)]
        try:
            for b, c in enumerate(saved):
                c2 = KpCfg.from_buffer_copy(c)
                c2.flags = c.flags & ~binding.FLAG_PDL   # other flags pick other kernels
                plan.set_config(b, M, c2)
            nopdl = _run(plan, x, wp, wfb, True, aux, evs)
        finally:
            for b, c in enumerate(saved):
                plan.set_config(b, M, c)
        for a, b in zip(seq, nopdl):
            assert torch.equal(a, b)
    finally:
        plan.set_overlap(-1)


# ---- F_B fused into the F_A/beta launch ------------------------------------------------------

FUSED_FAB = [KpCfg.make("tc05", split_k=C, k_unroll=nkb, stages=st,
                        flags=binding.FLAG_PDL | binding.FLAG_FUSE_FB)
             for (C, nkb, st) in ((1, 2, 0), (2, 4, 2), (4, 2, 3), (8, 4, 2), (16, 2, 0))]


@pytest.mark.parametrize("M", [1, 5, 16, 64, 128, 200])
@pytest.mark.parametrize("ci", range(len(FUSED_FAB)))
def test_kda_fused_fb(plan, M, ci):
    cf = FUSED_FAB[ci]
    saved = plan.get_config(binding.BRANCH_FAB, M)
    try:
        plan.set_config(binding.BRANCH_FAB, M, cf)
    except binding.KdaProjError as e:
        # no room for the F_B operands at this M, or more split-K scratch than
        # the plan holds
        assert e.code in (binding.KP_ECONFIG, binding.KP_ETOOBIG)
        pytest.skip(str(e))
    x, wp, wfb = kda_inputs(M, layer=3, seed=5)
    x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    try:
        seq = _run(plan, x, wp, wfb, False, aux, evs)
        ovl = _run(plan, x, wp, wfb, True, aux, evs)
        for a, b in zip(seq, ovl):
            assert torch.equal(a, b)
        check_kda(ovl, x.cpu(), wp.cpu(), wfb.cpu(), 4096, 136, f"fused C={cf.split_k} M={M}")
        # the fused F_B runs the same MMA sequence as the tcgen05 kernel with
        # one CTA per tile on the bf16 F_A: bit-identical
        ref_fb = binding.skinny_gemm(ovl[1][:, :128].contiguous(), wfb,
                                     cfg=KpCfg.make("tc05", split_k=1, k_unroll=2))
        torch.cuda.synchronize()
        assert torch.equal(ref_fb, ovl[2])
    finally:
        plan.set_config(binding.BRANCH_FAB, M, saved)
        plan.set_overlap(-1)


def test_kda_fused_fb_graph_replay(plan):
    M = 8
    cf = FUSED_FAB[3]
    saved = plan.get_config(binding.BRANCH_FAB, M)
    plan.set_config(binding.BRANCH_FAB, M, cf)
    x, wp, wfb = kda_inputs(M, layer=4, seed=6)
    x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    try:
        seq = _run(plan, x, wp, wfb, False, aux, evs)
        outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
        plan.set_overlap(1)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
        g.replay()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(seq, outs):
            assert torch.equal(a, b)
    finally:
        plan.set_config(binding.BRANCH_FAB, M, saved)
        plan.set_overlap(-1)


# ---- the whole projection as one launch (mode 2) -------------------------------------------

def _run_mode(plan, x, wp, wfb, mode, aux, evs):
    M = x.shape[0]
    outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
    plan.set_overlap(mode)
    plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
    torch.cuda.synchronize()
    return [o.clone() for o in outs]


@pytest.mark.parametrize("M", [1, 3, 16, 64, 128])
@pytest.mark.parametrize("C,nkb", [(4, 2), (8, 2), (16, 4)])
def test_kda_single_launch(plan, M, C, nkb):
    cq = KpCfg.make("tc05", split_k=C, k_unroll=nkb, stages=0)
    cf = KpCfg.make("tc05", split_k=C, k_unroll=nkb, stages=0)
    saved = [plan.get_config(b, M) for b in range(3)]
    try:
        try:
            plan.set_config(binding.BRANCH_QKVG, M, cq)
            plan.set_config(binding.BRANCH_FAB, M, cf)
        except binding.KdaProjError as e:
            pytest.skip(str(e))
        x, wp, wfb = kda_inputs(M, layer=6, seed=8)
        x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
        aux = torch.cuda.Stream()
        evs = binding.make_events()
        one = _run_mode(plan, x, wp, wfb, 2, aux, evs)
        check_kda(one, x.cpu(), wp.cpu(), wfb.cpu(), 4096, 136, f"single launch C={C} M={M}")
        seq = _run_mode(plan, x, wp, wfb, 0, aux, evs)
        # same split-K factor for both branches: identical to the sequential path
        assert torch.equal(one[0], seq[0]) and torch.equal(one[1], seq[1])
        # F_B: same MMA sequence as the tcgen05 kernel with one CTA per tile
        ref_fb = binding.skinny_gemm(one[1][:, :128].contiguous(), wfb,
                                     cfg=KpCfg.make("tc05", split_k=1, k_unroll=2))
        torch.cuda.synchronize()
        assert torch.equal(ref_fb, one[2])
        # captured and replayed
        outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
        plan.set_overlap(2)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(one, outs):
            assert torch.equal(a, b)
    finally:
        for b, c in enumerate(saved):
            plan.set_config(b, M, c)
        plan.set_overlap(-1)


CC_SINGLE = [KpCfg.make("cc", split_k=1, block=256, rows=2, k_unroll=4),   # 16 rows: cluster of 8
             KpCfg.make("cc", split_k=1, block=512, rows=1, k_unroll=4),   # 16 rows
             KpCfg.make("cc", split_k=1, block=256, rows=4, k_unroll=2),   # 32 rows: cluster of 4
             KpCfg.make("cc", split_k=1, block=128, rows=4, k_unroll=1)]   # 16 rows, 4 warps


def _single_launch_cc_check(p, M, cfg, K, Nq, Nfab, Nfb, layer, seed):
    x, wp, wfb = kda_inputs(M, layer=layer, seed=seed, K=K, Nq=Nq, Nfab=Nfab, Nfb=Nfb)
    xd, wpd, wfbd = x.cuda(), wp.cuda(), wfb.cuda()
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    p.set_config(binding.BRANCH_QKVG, M, cfg)
    assert p.overlap_at(M) in (0, 1, 2)
    outs = (poisoned((M, Nq)), poisoned((M, Nfab)), poisoned((M, Nfb)))
    p.set_overlap(2)
    p.run(xd, wpd, wfbd, *outs, aux_stream=aux, events=evs)
    torch.cuda.synchronize()
    check_kda(outs, x, wp, wfb, Nq, Nfab, f"CUDA-core single launch {cfg.as_dict()} M={M}")
    # each part equals the same CUDA-core kernel run on its own rows, and F_B
    # the small-K kernel (same k order) on the GPU's F_A
    q = binding.skinny_gemm(xd, wpd[:Nq].contiguous(), cfg=cfg)
    f = binding.skinny_gemm(xd, wpd[Nq:].contiguous(), cfg=cfg)
    b = binding.skinny_gemm(outs[1][:, :128].contiguous(), wfbd,
                            cfg=KpCfg.make("smallk", block=256, rows=16))
    torch.cuda.synchronize()
    assert torch.equal(q, outs[0]) and torch.equal(f, outs[1]) and torch.equal(b, outs[2])
    # captured and replayed
    again = (poisoned((M, Nq)), poisoned((M, Nfab)), poisoned((M, Nfb)))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        p.run(xd, wpd, wfbd, *again, aux_stream=aux, events=evs)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a_, b_ in zip(outs, again):
        assert torch.equal(a_, b_)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("ci", range(len(CC_SINGLE)))
def test_kda_single_launch_cuda_core(plan, M, ci):
    """Mode 2 with a one-slice CUDA-core Q/K/V/G configuration: one launch over
    the packed weight; the CTAs of the F_A rows form a cluster that computes
    F_B from the bf16 F_A it exchanges in distributed shared memory."""
    saved = [plan.get_config(b, M) for b in range(3)]
    try:
        _single_launch_cc_check(plan, M, CC_SINGLE[ci], 7168, 4096, 136, 1024, layer=9, seed=10)
    finally:
        for b, c in enumerate(saved):
            plan.set_config(b, M, c)
        plan.set_overlap(-1)


def test_kda_single_launch_cuda_core_ragged():
    """Ragged packed shape: the last tile of the F_A/beta rows is partly past
    N, whole padding CTAs leave at once, K = 1032 is not a multiple of the
    loop's step, and N_fb = 200 does not divide evenly over the cluster."""
    p = binding.KdaPlan(K=1032, N_qkvg=256, N_fab=136, N_fb=200, max_M=8)
    try:
        for M, cfg in ((1, CC_SINGLE[0]), (5, CC_SINGLE[1]), (8, CC_SINGLE[2]), (3, CC_SINGLE[3])):
            _single_launch_cc_check(p, M, cfg, 1032, 256, 136, 200, layer=2, seed=11)
    finally:
        p.close()


def test_single_launch_falls_back_for_a_cuda_core_config(plan):
    # 6 rows per CTA (3 warps x 2) do not tile the 128 F_A rows: no single-launch
    # form, so mode 2 runs the overlapped path
    M = 2
    saved = plan.get_config(binding.BRANCH_QKVG, M)
    try:
        plan.set_config(binding.BRANCH_QKVG, M, KpCfg.make("cc", split_k=1, block=96, rows=2,
                                                           k_unroll=4))
        x, wp, wfb = kda_inputs(M, layer=7, seed=9)
        outs = _run_mode(plan, x.cuda(), wp.cuda(), wfb.cuda(), 2, torch.cuda.Stream(),
                         binding.make_events())
        check_kda(outs, x, wp, wfb, 4096, 136, "mode 2 fallback")
    finally:
        plan.set_config(binding.BRANCH_QKVG, M, saved)
        plan.set_overlap(-1)


def test_plan_takes_any_split_within_its_reserve():
    """A plan reserves scratch for every tcgen05 split its branches' K allows
    at up to 256 tokens (F_B's K = 128: two K blocks, so a split of 2) and a
    combine ticket per output row, whatever its table entries need: a small
    plan accepts a 2-way tcgen05 F_B and a split-K CUDA-core Q/K/V/G
    configuration whose partials fit, and computes with them."""
    M = 4
    p = binding.KdaPlan(K=7168, N_qkvg=4096, N_fab=136, N_fb=1024, max_M=M)
    try:
        p.set_config(binding.BRANCH_FB, M, KpCfg.make("tc05", split_k=2, k_unroll=1))
        p.set_config(binding.BRANCH_QKVG, M, KpCfg.make("cc", split_k=4, block=256, rows=2, k_unroll=4))
        x, wp, wfb = kda_inputs(M, layer=3, seed=12)
        outs = _run_mode(p, x.cuda(), wp.cuda(), wfb.cuda(), 0, torch.cuda.Stream(), binding.make_events())
        check_kda(outs, x, wp, wfb, 4096, 136, "reserve-sized configs")
    finally:
        p.close()


# ---- boundary errors on a live device -------------------------------------------------------

def test_errors_on_device(plan):
    x, wp, wfb = kda_inputs(2, layer=0)
    x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
    # M above the plan's max_M
    big = torch.zeros((257, 7168), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.KdaProjError) as e:
        plan.run(big, wp, wfb)
    assert e.value.code == binding.KP_ETOOBIG
    # misaligned pointer (2-byte offset)
    flat = torch.zeros(2 * 7168 + 8, dtype=torch.bfloat16, device="cuda")
    xm = flat[1:1 + 2 * 7168].view(2, 7168)
    with pytest.raises(binding.KdaProjError) as e:
        binding.skinny_gemm(xm, wp[:64].contiguous())
    assert e.value.code == binding.KP_EALIGN
    # the CUDA-core kernel is for M <= 16
    with pytest.raises(binding.KdaProjError) as e:
        binding.skinny_gemm(torch.zeros((17, 7168), dtype=torch.bfloat16, device="cuda"),
                            wp[:64].contiguous(), cfg=KpCfg.make("cc", split_k=4, rows=1, k_unroll=4))
    assert e.value.code == binding.KP_ECONFIG
    # M = 0 leaves the outputs untouched
    empty = torch.zeros((0, 7168), dtype=torch.bfloat16, device="cuda")
    outs = (poisoned((0, 4096)), poisoned((0, 136)), poisoned((0, 1024)))
    plan.run(empty, wp, wfb, *outs)
    # a config needing more scratch than the plan holds is refused
    small = binding.KdaPlan(K=7168, N_qkvg=4096, N_fab=136, N_fb=1024, max_M=2)
    try:
        # 896 K slices of 8: 896 x 2 x 4232 fp32 partials, above the room for
        # a 16-way tcgen05 split at two tokens (16 x 16 x 128 fp32 per tile)
        cfg = KpCfg.make("cc", split_k=896, rows=1, k_unroll=4)
        with pytest.raises(binding.KdaProjError) as e:
            small.set_config(binding.BRANCH_QKVG, 2, cfg)
        assert e.value.code == binding.KP_ETOOBIG
    finally:
        small.close()


def test_repeat_calls_bit_identical():
    x, W = gemm_case(6, 4096, 7168, seed=11)
    x, W = x.cuda(), W.cuda()
    for cfg in (KpCfg.make("cc", split_k=7, rows=4, k_unroll=2),
                KpCfg.make("tc05", split_k=16, k_unroll=4)):
        a = binding.skinny_gemm(x, W, cfg=cfg)
        b = binding.skinny_gemm(x, W, cfg=cfg)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


def test_graph_keeps_its_scratch_after_the_workspace_grows():
    """skinny_gemm's per-device workspace grows on demand; the buffer it
    replaces stays allocated, so a graph captured before the growth still
    computes the same outputs when replayed after it."""
    M, N, K = 4, 4096, 7168
    x, W = gemm_case(M, N, K, seed=21)
    x, W = x.cuda(), W.cuda()
    cfg = KpCfg.make("tc05", split_k=8, k_unroll=2)   # partial tiles in the workspace
    ref = binding.skinny_gemm(x, W, cfg=cfg)
    torch.cuda.synchronize()
    y = poisoned((M, N))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.skinny_gemm(x, W, y, cfg=cfg)
    # 448 K slices x 16 tokens x 16384 rows of fp32 partial sums (470 MB):
    # more than any call before it needs, so the workspace grows
    xb = torch.zeros((16, K), dtype=torch.bfloat16, device="cuda")
    Wb = torch.zeros((16384, K), dtype=torch.bfloat16, device="cuda")
    binding.skinny_gemm(xb, Wb, cfg=KpCfg.make("cc", split_k=448, block=256, rows=4, k_unroll=1))
    torch.cuda.synchronize()
    del xb, Wb
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
