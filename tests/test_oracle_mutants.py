"""Each plausible mistake planted in a copy of the oracle's C source (on the
CPU, never on a GPU) must trip at least one pin; the pins are therefore not
just restating the oracle."""
import os
import tempfile

import pytest

import oracle
from oracle_pins import PINS

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()

MUTANTS = {
    "dropped_last_term": ("k < j->K; ++k", "k < j->K - 1; ++k"),
    "wrong_sign": ("acc = acc + p;", "acc = acc - p;"),
    "w_index_off_by_one": ("widen(wr[k], j->dtype)", "widen(wr[(k + 1) % j->K], j->dtype)"),
    "x_transposed": ("widen(xr[k], j->dtype)",
                     "widen(j->x[(int64_t)(k % j->M) * j->ldx + (m % j->K)], j->dtype)"),
    "float_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "round_half_away": ("double r = rint(ldexp(a, -qexp));", "double r = round(ldexp(a, -qexp));"),
    "round_truncate": ("double r = rint(ldexp(a, -qexp));", "double r = floor(ldexp(a, -qexp));"),
    "no_subnormal_quantum": ("int qexp = (E < -126) ? -133 : (E - 7);", "int qexp = E - 7;"),
    "widen_shift": ("((uint32_t)b) << 16", "((uint32_t)b) << 15"),
    "fa_truncated_not_rounded": (
        "fa_bf16[(int64_t)m * N_fa + j] = kdo_f64_to_bf16_rne(fab[(int64_t)m * N_fab + j]);",
        "{ float f_ = (float)fab[(int64_t)m * N_fab + j]; uint32_t u_; memcpy(&u_, &f_, 4);"
        " fa_bf16[(int64_t)m * N_fa + j] = (uint16_t)(u_ >> 16); }"),
    "fa_column_shift": ("kdo_f64_to_bf16_rne(fab[(int64_t)m * N_fab + j])",
                        "kdo_f64_to_bf16_rne(fab[(int64_t)m * N_fab + j + 1])"),
    "packed_slice_off_by_one": ("Wp + (int64_t)N_qkvg * K", "Wp + (int64_t)(N_qkvg - 1) * K"),
    "fb_reads_unrounded_width": ("fb, N_fb, M, N_fb, N_fa, nthreads", "fb, N_fb, M, N_fb, N_fa - 1, nthreads"),
    "fp16_exponent_bias": ("ldexp((double)(f | 0x400), e - 25)", "ldexp((double)(f | 0x400), e - 24)"),
    "fp16_subnormal_as_normal": ("v = ldexp((double)f, -24);", "v = ldexp((double)(f | 0x400), -25);"),
    "fp16_decoded_as_bf16": ("return dtype ? kdo_fp16_to_f64(b) : kdo_bf16_to_f64(b);",
                             "return kdo_bf16_to_f64(b);"),
    "residual_ignored": ("acc = acc + widen(j->res[(int64_t)m * j->ldr + n], j->dtype);", "acc = acc;"),
    "residual_doubled": ("acc = acc + widen(j->res[(int64_t)m * j->ldr + n], j->dtype);",
                         "acc = acc + 2.0 * widen(j->res[(int64_t)m * j->ldr + n], j->dtype);"),
    "residual_column_shift": ("widen(j->res[(int64_t)m * j->ldr + n], j->dtype)",
                              "widen(j->res[(int64_t)m * j->ldr + (n + 1) % j->N], j->dtype)"),
    "residual_row_shift": ("widen(j->res[(int64_t)m * j->ldr + n], j->dtype)",
                           "widen(j->res[(int64_t)((m + 1) % j->M) * j->ldr + n], j->dtype)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation anchor for {name} not unique"
    text = SRC.replace(old, new)
    with tempfile.TemporaryDirectory() as d:
        orc = oracle.Oracle.from_source(text, d)
        failed = []
        for pin in PINS:
            try:
                pin(orc)
            except AssertionError:
                failed.append(pin.__name__)
        assert failed, f"mutant {name} passed every pin"
