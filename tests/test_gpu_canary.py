"""Guard regions around every output: no kernel writes outside its output.

compute-sanitizer is not available here, so out-of-bounds stores are caught
the way a guard page would catch them: each output tensor is a view into a
larger allocation whose words before and after it hold a sentinel pattern,
and every kernel family, configuration kind and projection mode must leave
those words untouched. The interior is NaN-poisoned as in the parity tests,
so a missing store shows up too. A stray store lands in memory the test
owns, so it is reported rather than faulting.
"""
import pytest
import torch

from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.binding import KpCfg
from decode_projection_gemms_gb300.inputs import gen_w, gen_x

pytestmark = pytest.mark.gpu

PAD = 4096            # 16-bit words of guard on each side (8 KB; keeps 16-byte alignment)
SENTINEL = 0x5A5A     # a finite bf16/fp16 pattern no kernel here produces by accident
NAN16 = 0x7FC1        # bf16 NaN: the interior before the call


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_projection_gemms_gb300.build import build
    build()
    binding.load()
    binding.table_load()
    yield
    assert binding.device_error() == 0


class Guarded:
    """An [M, N] 16-bit output with PAD sentinel words before and after it."""

    def __init__(self, M, N, dtype=torch.bfloat16):
        self.M, self.N = M, N
        self.buf = torch.full((2 * PAD + M * N,), SENTINEL, dtype=torch.int16, device="cuda")
        self.buf[PAD:PAD + M * N] = NAN16
        self.t = self.buf[PAD:PAD + M * N].view(dtype).view(M, N)

    def check(self, label):
        torch.cuda.synchronize()
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.M * self.N:]
        bad_h = int((head != SENTINEL).sum())
        bad_t = int((tail != SENTINEL).sum())
        assert bad_h == 0 and bad_t == 0, f"{label}: {bad_h} words written before, {bad_t} after the output"
        inner = self.buf[PAD:PAD + self.M * self.N]
        assert int((inner == NAN16).sum()) == 0, f"{label}: output elements left unwritten"


GEMM_CONFIGS = [
    KpCfg.make("cc", split_k=1, block=256, rows=2, k_unroll=4),
    KpCfg.make("cc", split_k=3, block=128, rows=4, k_unroll=1),
    KpCfg.make("cc", split_k=1, block=224, rows=2, k_unroll=2, stages=4),
    KpCfg.make("cc", split_k=5, block=128, rows=1, k_unroll=4, stages=4),
    KpCfg.make("tc05", split_k=1, k_unroll=2),
    KpCfg.make("tc05", split_k=8, k_unroll=2, producers=2, stages=3),
    KpCfg.make("tc05", split_k=4, rows=256, k_unroll=1),
    None,   # the table's choice
]


@pytest.mark.parametrize("M", [1, 5, 16, 64, 300])
@pytest.mark.parametrize("N,K", [(136, 7168), (1000, 1032), (4096, 7168)])
@pytest.mark.parametrize("ci", range(len(GEMM_CONFIGS)))
def test_skinny_gemm_stays_inside_its_output(M, N, K, ci):
    cfg = GEMM_CONFIGS[ci]
    if cfg is not None:
        try:
            binding.scratch_bytes(M, N, K, cfg, 152)
        except binding.KdaProjError:
            pytest.skip("configuration not valid at this shape")
    x = gen_x(M, K, seed=M + 7).cuda()
    W = gen_w(N, K, seed=N + 3).cuda()
    y = Guarded(M, N)
    binding.skinny_gemm(x, W, y.t, cfg=cfg)
    y.check(f"skinny_gemm M={M} N={N} K={K} cfg={cfg.as_dict() if cfg else 'table'}")


@pytest.mark.parametrize("M", [1, 33])
def test_small_k_and_residual_stay_inside(M):
    K, N = 128, 1024
    x = gen_x(M, K, seed=2).cuda()
    W = gen_w(N, K, seed=4).cuda()
    y = Guarded(M, N)
    binding.skinny_gemm(x, W, y.t, cfg=KpCfg.make("smallk", block=256, rows=8))
    y.check(f"smallk M={M}")
    for dt in (torch.bfloat16, torch.float16):
        x2 = gen_x(M, 7168, seed=5, dtype=dt).cuda()
        W2 = gen_w(520, 7168, seed=6, dtype=dt).cuda()
        r = gen_x(M, 520, seed=8, dtype=dt).cuda()
        y2 = Guarded(M, 520, dt)
        binding.skinny_gemm_ex(x2, W2, r, y2.t)
        y2.check(f"skinny_gemm_ex {dt} M={M}")


@pytest.mark.parametrize("M", [1, 3, 16, 64, 128])
@pytest.mark.parametrize("mode", [0, 1, 2, -1])
def test_projection_stays_inside_its_outputs(M, mode):
    """Every mode of the projection (the table's choice included: the
    CUDA-core single launch at M = 1, the tcgen05 one above, the two-stream
    mode with F_B fused into the F_A/beta launch at M = 128)."""
    K, Nq, Nfab, Nfb = 7168, 4096, 136, 1024
    plan = binding.KdaPlan(K, Nq, Nfab, Nfb, max_M=128)
    try:
        x = gen_x(M, K, seed=M).cuda()
        wp = gen_w(Nq + Nfab, K, seed=11).cuda()
        wfb = gen_w(Nfb, 128, seed=12).cuda()
        outs = [Guarded(M, Nq), Guarded(M, Nfab), Guarded(M, Nfb)]
        plan.set_overlap(mode)
        plan.run(x, wp, wfb, *(o.t for o in outs), aux_stream=torch.cuda.Stream(), events=binding.make_events())
        for name, o in zip(("out_qkvg", "out_fab", "out_fb"), outs):
            o.check(f"projection M={M} mode={mode} {name}")
    finally:
        plan.set_overlap(-1)
        plan.close()
