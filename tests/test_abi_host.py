"""The C-ABI library without a GPU: it builds, loads, exports every function
``include/kdaproj.h`` declares, and its host-only logic (argument checks,
autotune-table parsing, configuration selection, scratch sizing) works."""
import ctypes
import os
import re
import subprocess

import pytest

from decode_projection_gemms_gb300 import binding
from decode_projection_gemms_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kdaproj.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^KP_API\s+(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("skinny_gemm", "kda_proj_plan", "kda_proj_run", "kda_proj_destroy",
                     "kp_last_error"):
        assert required in names
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, f"{name} not exported"
        getattr(lib, name)
    # internal symbols stay hidden
    assert not any(s.startswith("_ZN2kp") for s in exported)


def test_version_and_error_string(lib):
    assert lib.kp_version() == 1
    assert isinstance(lib.kp_last_error(), bytes)


def test_argument_errors_need_no_device(lib):
    p = ctypes.c_void_p(16)
    assert lib.skinny_gemm(p, p, p, 1, 8, 12, None, None) == binding.KP_ESHAPE     # K % 8
    assert b"multiple of 8" in lib.kp_last_error()
    assert lib.skinny_gemm(p, p, p, -1, 8, 16, None, None) == binding.KP_EINVAL
    assert lib.skinny_gemm(p, p, p, 0, 8, 16, None, None) == binding.KP_OK         # M = 0: no-op
    assert lib.skinny_gemm(None, p, p, 1, 8, 16, None, None) == binding.KP_EINVAL
    q = ctypes.c_void_p(24)
    assert lib.skinny_gemm(q, p, p, 1, 8, 16, None, None) == binding.KP_EALIGN
    assert lib.kda_proj_run(None, p, p, p, p, p, p, 1, None, None, None) == binding.KP_ENOPLAN
    out = ctypes.c_void_p()
    assert lib.kda_proj_plan(7168, 4096, 100, 1024, 16, ctypes.byref(out)) == binding.KP_ESHAPE
    assert lib.kda_proj_plan(7170, 4096, 136, 1024, 16, ctypes.byref(out)) == binding.KP_ESHAPE
    assert lib.kda_proj_plan(7168, 4096, 136, 1024, 0, ctypes.byref(out)) == binding.KP_EINVAL
    assert lib.kda_proj_destroy(None) == binding.KP_OK
    assert lib.kda_proj_set_overlap(None, 0) == binding.KP_ENOPLAN
    assert lib.kp_pdl_consumer_checksum(p, 4, None, 1, None) == binding.KP_EINVAL
    assert lib.kp_pdl_consumer_checksum(ctypes.c_void_p(17), 4, p, 1, None) == binding.KP_EALIGN
    assert lib.kp_selftest_timeout(0, None) == binding.KP_EINVAL
    assert lib.kp_selftest_timeout(2000000, None) == binding.KP_EINVAL
    # skinny_gemm_ex: element type and residual alignment, checked before any device work
    assert lib.skinny_gemm_ex(p, p, None, p, 1, 8, 16, 2, None, None) == binding.KP_EINVAL
    assert b"element type" in lib.kp_last_error()
    assert lib.skinny_gemm_ex(p, p, ctypes.c_void_p(17), p, 1, 8, 16, binding.DTYPE_FP16,
                              None, None) == binding.KP_EALIGN
    assert lib.skinny_gemm_ex(p, p, None, p, 1, 8, 12, binding.DTYPE_FP16, None, None) == binding.KP_ESHAPE
    assert lib.skinny_gemm_ex(p, p, p, p, 0, 8, 16, binding.DTYPE_FP16, None, None) == binding.KP_OK


def test_builtin_rule(lib):
    binding.table_clear()
    try:
        c = binding.select_config(1, 4096, 7168, num_sms=152)
        assert c.kind == binding.KIND_CC and c.split_k >= 1
        c = binding.select_config(64, 4096, 7168, num_sms=152)
        assert c.kind == binding.KIND_TC05
        c = binding.select_config(8, 1024, 128, num_sms=152)
        assert c.kind == binding.KIND_SMALLK
        # prefill: one launch, no split-K; 256-row CTAs once 128-row ones outnumber the SMs
        c = binding.select_config(1024, 4096, 7168, num_sms=152)
        assert (c.kind, c.split_k, c.rows, c.k_unroll) == (binding.KIND_TC05, 1, 0, 2)
        c = binding.select_config(4096, 4096, 7168, num_sms=152)
        assert (c.kind, c.split_k, c.rows, c.k_unroll) == (binding.KIND_TC05, 1, 256, 1)
    finally:
        binding.table_load()


def test_table_lookup_rounds_m_up(lib, tmp_path):
    t = tmp_path / "t.txt"
    t.write_text(
        "# M N K kind split_k block rows k_unroll producers stages flags overlap\n"
        "1 4096 7168 cc 7 256 4 2 0 0 1 1\n"
        "4 4096 7168 cc 5 128 2 4 0 0 1 1  # trailing comment\n"
        "16 4096 7168 tc05 4 0 0 2 2 3 1 0\n"
        "64 4096 7168 tc05 2 0 0 1 0 4 0 1\n")
    binding.table_load(str(t))
    try:
        assert binding.table_size() == 4
        c = binding.select_config(1, 4096, 7168, 152)
        assert (c.kind, c.split_k, c.block, c.rows, c.k_unroll) == (binding.KIND_CC, 7, 256, 4, 2)
        for M in (2, 3, 4):
            c = binding.select_config(M, 4096, 7168, 152)
            assert (c.kind, c.split_k, c.block, c.rows) == (binding.KIND_CC, 5, 128, 2)
        for M in (5, 9, 16):
            c = binding.select_config(M, 4096, 7168, 152)
            assert (c.kind, c.split_k, c.k_unroll, c.producers, c.stages) == (binding.KIND_TC05, 4, 2, 2, 3)
        c = binding.select_config(33, 4096, 7168, 152)
        assert (c.kind, c.split_k, c.k_unroll, c.stages, c.flags) == (binding.KIND_TC05, 2, 1, 4, 0)
        # beyond the largest bucket, or another (N, K): built-in rule
        c = binding.select_config(100, 4096, 7168, 152)
        assert c.kind == binding.KIND_TC05 and c.split_k == 4 and c.stages == 0
        c = binding.select_config(1, 4096, 1024, 152)
        assert c.kind == binding.KIND_CC
    finally:
        binding.table_load()


def test_shipped_table_entries_are_valid(lib):
    """Every entry of the shipped table names a configuration the library
    accepts for its shape (kernel built, shared memory and cluster limits),
    so no lookup hands a kernel a configuration it refuses. Entries with
    KP_FLAG_FUSE_FB belong to a plan's F_A/beta branch and are checked
    without the flag (the plan checks the fused form when it loads them)."""
    binding.table_load()
    assert binding.table_size() > 0
    n = 0
    for line in open(binding.TABLE_PATH):
        f = line.split("#")[0].split()
        if len(f) < 12:
            continue
        M, N, K = (int(v) for v in f[:3])
        cfg = binding.KpCfg.make(f[3], *(int(v) for v in f[4:11]))
        cfg.flags &= ~binding.FLAG_FUSE_FB
        binding.scratch_bytes(M, N, K, cfg, 152)   # raises KP_ECONFIG if refused
        n += 1
    assert n == binding.table_size()


def test_table_rejects_malformed(lib, tmp_path):
    t = tmp_path / "bad.txt"
    t.write_text("1 4096 7168 cc 7 256\n")
    with pytest.raises(binding.KdaProjError) as e:
        binding.table_load(str(t))
    assert e.value.code == binding.KP_EIO
    with pytest.raises(binding.KdaProjError):
        binding.table_load(str(tmp_path / "missing.txt"))
    binding.table_load()


def test_scratch_sizes(lib):
    cc = binding.KpCfg.make("cc", split_k=7, block=256, rows=4, k_unroll=2)
    # S x M x N fp32 partials + one counter per 32-row tile
    assert binding.scratch_bytes(4, 4096, 7168, cc, 152) == 7 * 4 * 4096 * 4 + (4096 // 32) * 4
    one = binding.KpCfg.make("cc", split_k=1, block=256, rows=4, k_unroll=2)
    assert binding.scratch_bytes(4, 4096, 7168, one, 152) == 0
    tc = binding.KpCfg.make("tc05", split_k=4, k_unroll=2, stages=3)
    # cluster split-K: C fp32 partial tiles of Mpad x 128 per feature tile
    # (M = 20 -> Mpad 32; N = 4096 -> 32 tiles)
    assert binding.scratch_bytes(20, 4096, 7168, tc, 152) == 32 * 4 * 32 * 128 * 4
    assert binding.scratch_bytes(20, 4096, 7168, binding.KpCfg.make("tc05", split_k=1), 152) == 0
    # token tiles of 256 beyond M = 256: one set of partial tiles per token tile
    tc_deep = binding.KpCfg.make("tc05", split_k=4, k_unroll=2, stages=0)
    assert binding.scratch_bytes(300, 4096, 7168, tc_deep, 152) == 2 * 32 * 4 * 256 * 128 * 4
    for bad_tc in (binding.KpCfg.make("tc05", split_k=3), binding.KpCfg.make("tc05", split_k=32),
                   binding.KpCfg.make("tc05", k_unroll=3), binding.KpCfg.make("tc05", stages=99),
                   binding.KpCfg.make("tc05", producers=6)):
        with pytest.raises(binding.KdaProjError):
            binding.scratch_bytes(20, 4096, 7168, bad_tc, 152)
    # 256 feature rows per CTA: partial tiles of Mpad x 256 fp32 (16 tiles)
    wide = binding.KpCfg.make("tc05", split_k=4, rows=256, k_unroll=1)
    assert binding.scratch_bytes(64, 4096, 7168, wide, 152) == 16 * 4 * 64 * 256 * 4
    with pytest.raises(binding.KdaProjError):   # a 256 KB stage does not fit
        binding.scratch_bytes(256, 4096, 7168, binding.KpCfg.make("tc05", split_k=4, rows=256,
                                                                  k_unroll=4), 152)
    bad = binding.KpCfg.make("cc", split_k=1, block=256, rows=8, k_unroll=1)
    with pytest.raises(binding.KdaProjError) as e:
        binding.scratch_bytes(16, 4096, 7168, bad, 152)     # 8 x 16 accumulators: not built
    assert e.value.code == binding.KP_ECONFIG


def test_split_k_partials_need_no_stage_memory(lib):
    # the partial tiles live in scratch, not in the pipeline's shared memory:
    # one stage is enough for any split factor, and only split_k > 1 has scratch
    def scratch(M, C, stages):
        return binding.scratch_bytes(M, 4096, 7168, binding.KpCfg.make(
            "tc05", split_k=C, k_unroll=1, stages=stages), 152)
    assert scratch(128, 4, 1) == 32 * 4 * 128 * 128 * 4
    assert scratch(128, 1, 1) == 0
    assert scratch(16, 16, 1) == 32 * 16 * 16 * 128 * 4


def test_fuse_flag_is_plan_only(lib):
    fused = binding.KpCfg.make("tc05", split_k=4, k_unroll=2,
                               flags=binding.FLAG_PDL | binding.FLAG_FUSE_FB)
    with pytest.raises(binding.KdaProjError) as e:
        binding.scratch_bytes(4, 136, 7168, fused, 152)
    assert e.value.code == binding.KP_ECONFIG


def test_missing_library_fails_loudly(tmp_path):
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(ImportError):
            binding.load(str(tmp_path / "nope.so"))
    finally:
        binding._lib = saved
