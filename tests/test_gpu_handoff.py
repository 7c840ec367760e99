"""Hand-off into a downstream kernel launched with programmatic dependent
launch: this library's kernels let dependents start early, and a dependent
that passes griddepcontrol.wait must see the projection's outputs complete,
in every mode, eagerly and in a captured graph. The consumer adds the 16-bit
patterns of each output exactly; outputs are NaN-poisoned first, so a read
that came too early would change the sum."""
import pytest
import torch

from decode_projection_gemms_gb300 import binding

from gpu_helpers import kda_inputs, poisoned

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    yield
    assert binding.device_error() == 0


@pytest.fixture(scope="module")
def plan():
    p = binding.KdaPlan(K=7168, N_qkvg=4096, N_fab=136, N_fb=1024, max_M=128)
    yield p
    p.close()


def bit_sum(t):
    return int(t.view(torch.int16).to(torch.int64).bitwise_and(0xFFFF).sum())


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("M", [1, 16, 128])
def test_pdl_consumer_sees_complete_outputs(plan, mode, M):
    x, wp, wfb = kda_inputs(M, layer=4, seed=3)
    x, wp, wfb = x.cuda(), wp.cuda(), wfb.cuda()
    aux = torch.cuda.Stream()
    evs = binding.make_events()
    outs = (poisoned((M, 4096)), poisoned((M, 136)), poisoned((M, 1024)))
    sums = torch.zeros(3, dtype=torch.int64, device="cuda")
    plan.set_overlap(mode)
    try:
        def step():
            sums.zero_()
            for o in outs:
                o.fill_(float("nan"))
            plan.run(x, wp, wfb, *outs, aux_stream=aux, events=evs)
            for i, o in enumerate(outs):
                binding.pdl_consumer_checksum(o, sums[i:i + 1])
        step()
        torch.cuda.synchronize()
        expect = [bit_sum(o) for o in outs]
        assert sums.tolist() == expect
        assert all(not torch.isnan(o.float()).any() for o in outs)
        # the same inside a captured graph, replayed twice
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(2):
            g.replay()
            torch.cuda.synchronize()
            assert sums.tolist() == expect
    finally:
        plan.set_overlap(-1)
