"""skinny_gemm_noalloc, called through the C ABI, must give what skinny_gemm
gives for the same inputs, on two calls in a row.

skinny_gemm_noalloc is for callers that cannot allocate device memory
(processes whose memory belongs to a pooling allocator, paths that cannot take
cudaMalloc's synchronisation): its split-K
partial sums live in a fixed device array inside the library. The second call
checks that the shared array (tickets left at zero, partial sums overwritten)
serves a new call correctly. This file sorts last so a run that stops at the
first failure has already run every other test; it also passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg
from decode_projection_gemms_gb300.inputs import bf16_bits, gen_w, gen_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    return binding.load()


def _noalloc(lib, x, W, y, cfg):
    M, K = x.shape
    N = W.shape[0]
    return lib.skinny_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                   ctypes.c_void_p(y.data_ptr()), M, N, K,
                                   ctypes.byref(cfg) if cfg is not None else None,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # (M, N, K, explicit CUDA-core config or None for the entry point's own choice)
    (1, 4096, 7168, None),
    (4, 136, 7168, None),
    (3, 1000, 2048, KpCfg.make("cc", split_k=8, block=256, rows=2, k_unroll=2)),
    (16, 1024, 7168, KpCfg.make("cc", split_k=7, block=256, rows=4, k_unroll=1)),
]


@pytest.mark.parametrize("M,N,K,cfg", CASES)
def test_noalloc_matches_skinny_gemm_twice(lib, M, N, K, cfg):
    x = gen_x(M, K, seed=31 + M).cuda()
    W = gen_w(N, K, seed=37 + M).cuda()
    ref_cfg = cfg if cfg is not None else KpCfg.make("cc", split_k=4, block=256, rows=4, k_unroll=2)
    ref = binding.skinny_gemm(x, W, cfg=ref_cfg)           # the existing entry point
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    exact = oracle.gemm(bf16_bits(x.cpu()), bf16_bits(W.cpu()))
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(lib, x, W, y, cfg)
        assert rc == binding.KP_OK, lib.kp_last_error().decode()
        torch.cuda.synchronize()
        got = y.float().cpu().numpy().astype(np.float64)
        r = oracle.compare(got, ref64)                        # same tolerance as the parity tests
        assert r["ok"], f"call {call}: {r}"
        assert oracle.compare(got, exact)["ok"]
        if cfg is not None:                                   # same kernel and configuration
            assert torch.equal(y, ref)


def test_noalloc_rejects_what_does_not_fit(lib):
    x = gen_x(16, 7168, seed=1).cuda()
    W = gen_w(8192, 7168, seed=2).cuda()
    y = torch.empty((16, 8192), dtype=torch.bfloat16, device="cuda")
    too_many_slices = KpCfg.make("cc", split_k=28, block=256, rows=4, k_unroll=1)
    assert _noalloc(lib, x, W, y, too_many_slices) == binding.KP_ETOOBIG
    assert b"fixed scratch" in lib.kp_last_error()
    # the entry point's own choice cannot fit either: x's slice (16 x 16384
    # 16-bit elements) needs split_k >= 3 to fit in 200 KiB of shared memory,
    # and 3 * 16 * 16384 partial sums exceed the array
    xk = gen_x(16, 16384, seed=4).cuda()
    Wk = torch.zeros((16384, 16384), dtype=torch.bfloat16, device="cuda")
    yk = torch.empty((16, 16384), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, xk, Wk, yk, None) == binding.KP_ETOOBIG
    del Wk
    x17 = gen_x(17, 7168, seed=3).cuda()
    y17 = torch.empty((17, 8192), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, x17, W, y17, None) == binding.KP_ECONFIG
    assert _noalloc(lib, x, W, y, KpCfg.make("tc05", split_k=4)) == binding.KP_ECONFIG


def test_noalloc_reads_a_w_written_by_the_kernel_before_it(lib):
    """With cfg NULL there is no programmatic dependent launch: a W that the
    previous kernel on the stream (here skinny_gemm, whose kernels let their
    dependents start before they store) has just written is read complete."""
    M, K1, N1 = 8, 2048, 1024   # first call: T = bf16(x1 @ W1^T), [8, 1024]
    x1 = gen_x(M, K1, seed=51).cuda()
    W1 = gen_w(N1, K1, seed=52, std=0.5).cuda()
    x2 = gen_x(4, N1, seed=53).cuda()   # second call: y = bf16(x2 @ T^T), W = T
    for _ in range(2):
        T = torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")
        y = torch.full((4, M), float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.skinny_gemm(x1, W1, T)                       # the table's choice, with PDL
        rc = _noalloc(lib, x2, T, y, None)
        assert rc == binding.KP_OK, lib.kp_last_error().decode()
        torch.cuda.synchronize()
        ref = oracle.gemm(bf16_bits(x2.cpu()), bf16_bits(T.cpu()))
        r = oracle.compare(y.float().cpu().numpy().astype(np.float64), ref)
        assert r["ok"], r
