"""The failure path on the GPU, without a fault: a kernel wait that nothing
completes must give up after its limit, report a code through the device
error word and leave the context usable (no trap, no hang)."""
import time

import pytest
import torch

from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg

from gpu_helpers import check_gemm, gemm_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    assert binding.device_error() == 0


def test_wait_runs_out_and_reports():
    t0 = time.perf_counter()
    binding.selftest_timeout(2000)        # 2 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert binding.device_error() == binding.DEV_SELFTEST
    assert binding.device_error() == 0    # read and cleared
    assert elapsed < 5.0
    # the context is still usable: a GEMM afterwards is correct
    x, W = gemm_case(3, 520, 2048, seed=1)
    check_gemm(x, W, KpCfg.make("tc05", split_k=4, k_unroll=2), "after the self-test")
    assert binding.device_error() == 0


def test_give_up_is_refused_until_read():
    """After a wait ran out, the entry points refuse new work (KP_EDEVICE, a
    host-visible error without a synchronising call) until kp_device_error()
    has read and cleared the code; then they run again."""
    binding.selftest_timeout(1000)
    torch.cuda.synchronize()
    x, W = gemm_case(2, 264, 1024, seed=3)
    x, W = x.cuda(), W.cuda()
    with pytest.raises(binding.KdaProjError) as e:
        binding.skinny_gemm(x, W)
    assert e.value.code == binding.KP_EDEVICE
    plan = binding.KdaPlan(K=1024, N_qkvg=256, N_fab=136, N_fb=64, max_M=4)
    try:
        wp = torch.zeros((392, 1024), dtype=torch.bfloat16, device="cuda")
        wfb = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(binding.KdaProjError) as e:
            plan.run(x, wp, wfb)
        assert e.value.code == binding.KP_EDEVICE
        assert binding.device_error() == binding.DEV_SELFTEST
        plan.run(x, wp, wfb)                  # accepted again
        torch.cuda.synchronize()
    finally:
        plan.close()
    check_gemm(x.cpu(), W.cpu(), None, "after reading the code")
    # the binding's checked run raises on a give-up during the call itself
    binding.selftest_timeout(1000)
    with pytest.raises(binding.KdaProjError) as e:
        binding.check_device()
    assert e.value.code == binding.KP_EDEVICE
    assert binding.device_error() == 0


def test_first_code_wins_and_streams_keep_order():
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.selftest_timeout(1000, stream=s)
        binding.selftest_timeout(1000, stream=s)
    s.synchronize()
    assert binding.device_error() == binding.DEV_SELFTEST
    assert binding.device_error() == 0
