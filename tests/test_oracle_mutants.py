"""Planted mistakes in the oracle must be caught by its pins.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong index, a wrong sign, a wrong rounding rule, a skipped
destination), builds it with gcc into a temporary directory and checks that
at least one pin of tests/oracle_pins.py fails.  The mistakes are planted in
the oracle on the CPU only; no GPU code is involved.
"""
import os
import subprocess

import pytest

import oracle as oracle_mod
from tests.oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle_mod.__file__), "gg_oracle.c")

MUTANTS = {
    "block_index_by_destination": ("int64_t dst = out_off + ((i * M + m) * ld_out + n) * esize;",
                                   "int64_t dst = out_off + ((q * M + m) * ld_out + n) * esize;"),
    "columns_reversed": ("src + (m * ld_in + n) * esize", "src + (m * ld_in + (N - 1 - n)) * esize"),
    "local_copy_skipped": ("for (int q = 0; q < world_size; ++q)", "for (int q = 1; q < world_size; ++q)"),
    "member_off_by_one": ("if (rank_start + i * rank_stride == h)", "if (rank_start + i * rank_stride == h + 1)"),
    "group_stride_ignored": ("int d = rank_start + q * rank_stride;", "int d = rank_start + q;"),
    "dropped_first_k": ("for (int64_t k = 0; k < K; ++k)\n                    s += a[k] * b[k];",
                        "for (int64_t k = 1; k < K; ++k)\n                    s += a[k] * b[k];"),
    "wrong_sign_sum": ("s += a[k] * b[k];", "s -= a[k] * b[k];"),
    "b_transposed_pitch": ("bt[n * K + k] = oracle_decode16(B[k * ldb + n], fmt);",
                           "bt[n * K + k] = oracle_decode16(B[(k % N) * ldb + (n % K)], fmt);"),
    "a2a_source_block_swapped": ("int64_t from = ((d * M + m) * ld_in + n) * esize;",
                                 "int64_t from = ((i * M + m) * ld_in + n) * esize;"),
    "a2a_dest_block_swapped": ("int64_t to = ((i * M + m) * ld_out + n) * esize;",
                               "int64_t to = ((d * M + m) * ld_out + n) * esize;"),
    "b_column_shifted": ("B[k * ldb + n]", "B[k * ldb + (n + 1) % N]"),
    "a_row_shifted": ("A[m * lda + k]", "A[((m + 1) % M) * lda + k]"),
    "decode_bias_off_by_one": ("v = ldexp((double)((1 << mbits) + f), e - bias - mbits);",
                               "v = ldexp((double)((1 << mbits) + f), e - bias - mbits + 1);"),
    "ties_away_from_zero": ("return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;", "return fl + 1.0;"),
    "no_subnormal_clamp": ("    if (e < emin)\n        e = emin;", ""),
    "bf16_mantissa_width": ("*ebits = 8; *mbits = 7;  *bias = 127;", "*ebits = 8; *mbits = 7;  *bias = 126;"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, source, name):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "gg_oracle.c"
    src.write_text(source.replace(old, new))
    lib_path = str(tmp_path / f"libgg_oracle_{name}.so")
    subprocess.run(["gcc", *oracle_mod._CFLAGS, "-o", lib_path, str(src), "-lm"], check=True)
    mutant = oracle_mod.Oracle(oracle_mod.load(lib_path))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
