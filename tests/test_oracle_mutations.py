"""Planted mistakes in the oracle must fail its pins (no GPU).

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong sign, a wrong scale, a transposed index, a wrong
rounding), builds it, and runs every pin against it in a child process.  The
pins must reject every mutant; the unmodified source must pass them.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "split_scale_wrong": ("float r1 = (a - a0) * 256.0f;", "float r1 = (a - a0) * 128.0f;"),
    "split_third_component_dropped": ("float a2 = (r1 - a1) * 256.0f;", "float a2 = (r1 - a1) * 0.0f;"),
    "split_rounds_to_nearest": ("return float_of(bits_of(x) & 0xFFFF0000u);",
                                "return float_of((bits_of(x) + 0x8000u) & 0xFFFF0000u);"),
    "band4_dropped": ("for (int band = 0; band <= 4; ++band)", "for (int band = 0; band <= 3; ++band)"),
    "band1_sign": ("acc = acc + S[1] * band_scale[1];", "acc = acc - S[1] * band_scale[1];"),
    "band2_scale": ("0x1p-16f, 0x1p-24f", "0x1p-15f, 0x1p-24f"),
    "one_acc_band_misplaced": ("int j = band - i;\n                            if (j < 0 || j > 2) continue;\n                            float p",
                               "int j = (band + 1) % 5 - i;\n                            if (j < 0 || j > 2) continue;\n                            float p"),
    "tf32_hi_lo_dropped": ("acc = acc + p_hl;", ";"),
    "tf32_lo_times_lo_added": ("acc = acc + p_hh;", "acc = acc + p_hh; acc = acc + alo[k] * blo[k];"),
    "tf32_ties_away": ("u += 0x00000FFFu + keep_lsb;", "u += 0x00001000u;"),
    "opB_transposed_index": ("p[n * K + k] = transB ? B[n * ldb + k] : B[k * ldb + n];",
                             "p[n * K + k] = transB ? B[k * ldb + n] : B[n * ldb + k];"),
    "opA_transposed_index": ("p[m * K + k] = transA ? A[k * lda + m] : A[m * lda + k];",
                             "p[m * K + k] = transA ? A[m * lda + k] : A[k * lda + m];"),
    "f64_beta_sign": ("if (beta != 0.0) c += beta * (double)Cold[m * ldc + n];",
                      "if (beta != 0.0) c -= beta * (double)Cold[m * ldc + n];"),
    "f64_product_in_float": ("s += (double)ar[k] * (double)br[k];",
                             "s += (double)(float)((double)ar[k] * (double)br[k]);"),
    "sgemm_first_term_dropped": ("acc = fmaf(ar[k], br[k], acc);",
                                 "acc = (k == 0) ? 0.0f : fmaf(ar[k], br[k], acc);"),
    "sgemm_unfused": ("acc = fmaf(ar[k], br[k], acc);",
                      "acc = acc + (float)((double)ar[k] * (double)br[k]);"),
    "sgemm_descending_k": ("for (int64_t k = 0; k < K; ++k) acc = fmaf(ar[k], br[k], acc);",
                           "for (int64_t k = K - 1; k >= 0; --k) acc = fmaf(ar[k], br[k], acc);"),
    "bias_dropped": ("if (bias_elem) c = c + *bias_elem;", ";"),
    "bf16x6_band1_scale": ("            acc = acc + S[1] * 0x1p-8f;\n            acc = acc + S[0];",
                           "            acc = acc + S[1] * 0x1p-7f;\n            acc = acc + S[0];"),
    "tf32x1_truncates": ("for (int64_t i = 0; i < M * K; ++i) pa[i] = tf32_rn(pa[i]);",
                         "for (int64_t i = 0; i < M * K; ++i) pa[i] = tf32_rz(pa[i]);"),
    # tensor-core model
    "tc_aligns_on_product_exponent": ("const int e = ilogb((double)a[i]) + ilogb((double)b[i]);",
                                      "const int e = ilogb((double)a[i] * (double)b[i]);"),
    "tc_three_alignment_bits": ("const int q = emax - 23 - neab;", "const int q = emax - 24 - neab;"),
    "tc_rounds_to_nearest": ("if (round_mode == 0 && fabs((double)f) > fabs(v))",
                             "if (round_mode == 7 && fabs((double)f) > fabs(v))"),
    "tc_floors_terms": ("S += (int64_t)trunc(ldexp((double)a[i] * (double)b[i], -q));",
                        "S += (int64_t)floor(ldexp((double)a[i] * (double)b[i], -q));"),
    "tc_issue_largest_first": ("pi9[9] = {2, 1, 2, 0, 1, 2, 0, 1, 0}, pj9[9] = {2, 2, 1, 2, 1, 0, 1, 0, 0}",
                               "pi9[9] = {0, 1, 0, 2, 1, 0, 2, 1, 2}, pj9[9] = {0, 0, 1, 0, 1, 2, 1, 2, 2}"),
    "tc_stage_doubled": ("    if (block < 1 || block > 64 || stage_k < block",
                         "    stage_k *= 2;\n    if (block < 1 || block > 64 || stage_k < block"),
    # exact-accumulation reference
    "exact_band3_product_dropped": ("sa_add(&s, a2 * b1 * 0x1p-24);", ";"),
    "exact_band1_scale": ("sa_add(&s, a0 * b1 * 0x1p-8);", "sa_add(&s, a0 * b1 * 0x1p-7);"),
    "exact_tf32_lo_hi_dropped": ("sa_add(&s, a0 * b1);\n                        sa_add(&s, a1 * b0);",
                                 "sa_add(&s, a0 * b1);"),
    "exact_no_sticky_bit": ("if (sticky) t53 |= 1u;", ";"),
    "exact_sign_ignored": ("const int64_t sg = (u >> 63) ? -1 : 1;", "const int64_t sg = 1;"),
    "exact_carry_truncates": ("const int64_t c = (s->d[i] - (s->d[i] & 0xFFFFFFFF)) / ((int64_t)1 << 32);",
                              "const int64_t c = s->d[i] / ((int64_t)1 << 32);"),
    "tc_owner_last": ("acc = part[owner];\n                for (int q = 0; q < pieces; ++q)\n                    if (q != owner) acc = acc + part[q];",
                      "acc = part[owner == 0 ? 1 : 0];\n                for (int q = 0; q < pieces; ++q)\n                    if (q != (owner == 0 ? 1 : 0)) acc = acc + part[q];"),
}


def _run(so_path):
    env = dict(os.environ, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "tests._mutant_runner", so_path], cwd=ROOT,
                          env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_oracle_passes_reduced_pins(tmp_path):
    so = oracle.build_variant(oracle.source(), str(tmp_path / "orig.so"))
    r = _run(so)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    so = oracle.build_variant(src.replace(old, new), str(tmp_path / f"{name}.so"))
    r = _run(so)
    assert r.returncode != 0, f"mutant {name} passed every pin"
