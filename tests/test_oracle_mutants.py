"""Plant plausible mistakes in a copy of oracle.c and check that a pin catches each.

Each mutant is compiled with the same flags as the real oracle into a temporary
directory and the pins of oracle_pins.py run against it in a child process
(so a mutant that reads out of bounds cannot take the test run down).  The
test passes only if every mutant fails at least one pin.
"""
import os
import subprocess
import sys
import textwrap

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("dropped_last_k_term", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    ("c_term_wrong_sign", "r += beta * (double)C[i * ldc + j];", "r -= beta * (double)C[i * ldc + j];"),
    ("c_index_transposed", "r += beta * (double)C[i * ldc + j];", "r += beta * (double)C[j * ldc + i];"),
    ("alpha_dropped", "double r = alpha * sum;", "double r = sum;"),
    ("alpha_on_c_too", "r += beta * (double)C[i * ldc + j];", "r += alpha * beta * (double)C[i * ldc + j];"),
    ("b_not_transposed", "double b = val[brow[k]];", "double b = val[B[k * ldb + j]];"),
    ("a_row_stride_ignored", "    return A + i * lda;", "    return A + i;"),
    ("gather_index_ignored", "    return A + r * lda;", "    return A + i * lda;"),
    ("gather_no_range_check", "if (r < 0 || r >= table_rows)", "if (r < 0)"),
    ("f16_bias_off_by_one", "e - 25);", "e - 24);"),
    ("f16_subnormal_scale", "ldexp((double)f, -24);", "ldexp((double)f, -25);"),
    ("bf16_fraction_width", "(f | 0x80), e - 134)", "(f | 0x80), e - 133)"),
    ("bf16_treated_as_f16", "const double *val = g_value[dtype == ORACLE_BF16 ? ORACLE_BF16 : ORACLE_F16];",
     "const double *val = g_value[ORACLE_F16];"),
    ("abs_not_absolute", "sum_abs += fabs(a) * fabs(b);", "sum_abs += a * b;"),
    ("beta_zero_reads_c", "if (C && beta != 0.0)", "if (C)"),
    ("scatter_c_row_from_source", "r += beta * (double)C[d * ldc + j];",
     "r += beta * (double)C[i * ldc + j];"),
    ("scatter_a_row_from_destination", "const uint16_t *arow = A + i * lda;\n        double *out",
     "const uint16_t *arow = A + d * lda;\n        double *out"),
    ("scatter_no_range_check", "if (d < 0 || d >= d_rows)", "if (d < 0)"),
    ("scatter_b_row_fixed", "const uint16_t *brow = B + j * ldb;\n            double sum",
     "const uint16_t *brow = B;\n            double sum"),
    ("fp4_nibble_order_swapped", "int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);",
     "int code = (k % 2 == 0) ? (byte >> 4) : (byte & 15);"),
    ("fp4_scale_block_16", "Ws[(k / 32) * lds + j]", "Ws[(k / 16) * lds + j]"),
    ("fp4_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("fp4_subnormal_value", "e == 0 ? 0.5 * m :", "e == 0 ? 1.0 * m :"),
    ("fp4_sign_ignored", "    return sign ? -v : v;\n}\n\ndouble oracle_decode_ue8m0",
     "    return v;\n}\n\ndouble oracle_decode_ue8m0"),
    ("ue8m0_bias", "ldexp(1.0, s - 127)", "ldexp(1.0, s - 128)"),
    ("fp4_scale_transposed", "Ws[(k / 32) * lds + j]", "Ws[j * lds + (k / 32)]"),
    # (swapping the nibble order of both FP4 operands alike permutes K the same
    # way on both sides, within a 32-element block: the products are unchanged,
    # so that mistake cannot be told apart and is not planted; the order is
    # pinned where an FP4 operand meets a 16-bit one)
    ("e2m1_scale_block_16", "scales[(k / 32) * lds + row]", "scales[(k / 16) * lds + row]"),
    ("e2m1_scale_transposed", "scales[(k / 32) * lds + row]", "scales[row * lds + (k / 32)]"),
    ("e2m1_a_scaled_by_b_scales", "fp4_element(arow, As, ldas, i, k)", "fp4_element(arow, Bs, ldbs, i, k)"),
    ("e2m1_a_scale_of_b_row", "fp4_element(arow, As, ldas, i, k)", "fp4_element(arow, As, ldas, 0, k)"),
    ("e2m1_b_row_stride_ignored", "const uint8_t *brow = Bq + j * ldbq;", "const uint8_t *brow = Bq + j;"),
    ("e2m1_a_row_stride_ignored", "const uint8_t *arow = Aq + i * ldaq;", "const uint8_t *arow = Aq + i;"),
    ("e2m1_alpha_dropped", "double d = alpha * dot;", "double d = dot;"),
    ("e2m1_c_wrong_sign", "d += beta * (double)C[i * ldc + j];", "d -= beta * (double)C[i * ldc + j];"),
    ("e2m1_last_k_dropped", "for (int64_t k = 0; k < K; ++k) {\n                double a = fp4_element",
     "for (int64_t k = 0; k + 1 < K; ++k) {\n                double a = fp4_element"),
    ("sign_bit_ignored_f16", "    return sign ? -v : v;\n}\n\n/* bfloat16", "    return v;\n}\n\n/* bfloat16"),
]

RUNNER = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import oracle, oracle_pins
    oracle.load({lib!r})
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except Exception as e:
            failed.append(pin.__name__)
    print("FAILED_PINS=" + ",".join(failed))
""")


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, bad):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(orig, bad, 1)
    csrc = tmp_path / "oracle_mutant.c"
    csrc.write_text(mutated)
    lib = str(tmp_path / "liboracle_mutant.so")
    oracle.build(str(csrc), lib)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED_PINS=")]
    if not line:
        # the mutant crashed the child (e.g. read out of bounds): caught.
        assert r.returncode != 0
        return
    failed = line[0].split("=", 1)[1]
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness on an unmodified copy reports no failing pin."""
    lib = str(tmp_path / "liboracle_copy.so")
    oracle.build(SRC, lib)
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    assert "FAILED_PINS=\n" in r.stdout + "\n" or r.stdout.strip().endswith("FAILED_PINS="), r.stdout + r.stderr
