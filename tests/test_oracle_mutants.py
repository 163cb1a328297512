"""Plant plausible mistakes in copies of the oracle and check the pins catch each.

Each mutant is the oracle's C source with one edit (a dropped term, a wrong sign
or index, a transposed operand, a float accumulator, ...).  A copy is compiled
into a temporary directory with the oracle's own flags and every pin is run on
it; at least one pin must fail.  The real oracle is untouched.
"""
import json
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle_gemm.c")

ROW_LOOP = "for (int64_t k = 0; k < jb->K; ++k) {\n        const double a = (double)arow[k];"
MUTANTS = {
    "drop_last_term": (ROW_LOOP, ROW_LOOP.replace("k < jb->K", "k + 1 < jb->K")),
    "skip_first_term": (ROW_LOOP, ROW_LOOP.replace("int64_t k = 0", "int64_t k = 1")),
    "wrong_sign": ("crow[j] += a * (double)bk[j];", "crow[j] -= a * (double)bk[j];"),
    "transposed_B": ("crow[j] += a * (double)bk[j];", "crow[j] += a * (double)jb->B[j * jb->ldb + k];"),
    "transposed_A": ("const double a = (double)arow[k];", "const double a = (double)jb->A[k * jb->lda + i];"),
    "ignores_lda": ("const float *arow = jb->A + i * jb->lda;", "const float *arow = jb->A + i * jb->K;"),
    "ignores_ldb": ("const float *bk = jb->B + k * jb->ldb;", "const float *bk = jb->B + k * jb->N;"),
    "float_accumulator": ("crow[j] += a * (double)bk[j];", "crow[j] = (float)(crow[j] + a * (double)bk[j]);"),
    "float_product": ("crow[j] += a * (double)bk[j];", "crow[j] += (double)((float)a * (float)bk[j]);"),
    "last_column_dropped": ("for (int64_t j = 0; j < jb->N; ++j) crow[j] += a",
                            "for (int64_t j = 0; j + 1 < jb->N; ++j) crow[j] += a"),
    "signed_bound": ("const double aa = fabs(a);", "const double aa = a;"),
    "bound_missing_b": ("brow[j] += aa * fabs((double)bk[j]);", "brow[j] += aa;"),
    "off_by_one_row": ("const int64_t i = jb->rows ? jb->rows[r] : r;\n    double *crow",
                       "const int64_t i = jb->rows ? jb->rows[r] : (r > 0 ? r - 1 : 0);\n    double *crow"),
    # general form
    "general_transa_ignored": ("jb->transa ? jb->A[k * jb->lda + i] : jb->A[i * jb->lda + k]",
                               "jb->A[i * jb->lda + k]"),
    "general_transb_wrong_index": ("jb->transb ? jb->B[j * jb->ldb + k]", "jb->transb ? jb->B[k * jb->ldb + j]"),
    "general_beta_dropped": ("            v += beta * c;", "            v += 0.0 * c;"),
    "general_alpha_dropped": ("double v = alpha * out[j];", "double v = out[j];"),
    "general_alpha_on_c": ("            v += beta * c;", "            v += alpha * beta * c;"),
    "general_reads_c_when_beta_zero": ("if (jb->beta != 0.0f) { /* beta == 0: C_in is not read */",
                                       "if (jb->Cin) {"),
    "general_bound_ignores_c": ("vb += fabs(beta) * fabs(c);", "vb += 0.0;"),
    "general_rows_ignored": ("const int64_t i = jb->rows ? jb->rows[r] : r;\n    double *out",
                             "const int64_t i = r;\n    double *out"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    so = oracle.compile_source(str(src), str(tmp_path / "libmutant.so"))
    # A mutant may read out of bounds and crash, so the pins run in a child
    # process; a crash counts as caught.
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import json, sys\n"
        f"sys.path[:0] = [{here!r}, {os.path.dirname(here)!r}]\n"
        "import oracle\n"
        "from oracle_pins import ALL_PINS\n"
        f"lib = oracle.OracleLib({so!r})\n"
        "failed = []\n"
        "for pin in ALL_PINS:\n"
        "    try:\n"
        "        pin(lib)\n"
        "    except Exception as e:\n"
        "        failed.append(pin.__name__ + ':' + type(e).__name__)\n"
        "print(json.dumps(failed))\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return  # crashed: caught
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"no pin caught mutant {name}"
