"""The oracle's pins catch plausible mistakes: each case below plants one mistake in a copy
of the oracle (its C source or its Python side), rebuilds that copy on the CPU and runs the
oracle's pin tests against it, which must then fail.  The mistakes are the kinds the pins are
meant to catch: a wrong or transposed index, a dropped term, a wrong zero point or group, a
wrong activation constant, a wrong mask.

Opt in with ``-m slow`` (each case rebuilds the oracle and runs the pins, ~10 s)."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PIN_TESTS = ["tests/test_oracle_pins.py", "tests/test_oracle_epilogue.py",
             "tests/test_oracle_dequant.py", "tests/test_oracle_backward.py"]

MUTANTS = {
    "B column index ignores the selected columns": (
        "tg_oracle.c",
        "Bsel[k * nc + c] = (float)tg_oracle_f16_to_f64(B[k * ldb + cols[c]]);",
        "Bsel[k * nc + c] = (float)tg_oracle_f16_to_f64(B[k * ldb + c]);"),
    "A row index ignores the selected rows": (
        "tg_oracle.c",
        "const uint16_t* arow = A + rows[r] * lda;",
        "const uint16_t* arow = A + r * lda;"),
    "B read transposed": (
        "tg_oracle.c",
        "Bsel[k * nc + c] = (float)tg_oracle_f16_to_f64(B[k * ldb + cols[c]]);",
        "Bsel[k * nc + c] = (float)tg_oracle_f16_to_f64(B[cols[c] * ldb + k]);"),
    "last k term dropped": (
        "tg_oracle.c",
        "      for (int64_t k = 0; k < K; ++k) {\n        float a =",
        "      for (int64_t k = 0; k + 1 < K; ++k) {\n        float a ="),
    "int4 zero point 7 instead of 8": (
        "tg_oracle.c",
        "tg_oracle_f64_to_f16((double)(q - 8) * s)",
        "tg_oracle_f64_to_f16((double)(q - 7) * s)"),
    "int4 nibble order reversed": (
        "tg_oracle.c",
        "(word >> (4 * (n % 8))) & 0xFu",
        "(word >> (4 * (7 - n % 8))) & 0xFu"),
    "int4 scale group of half the rows": (
        "tg_oracle.c",
        "scales[(k / group) * lds + n]",
        "scales[(k / (group > 1 ? group / 2 : 1)) * lds + n]"),
    "int4 scale of the next column": (
        "tg_oracle.c",
        "scales[(k / group) * lds + n]",
        "scales[(k / group) * lds + (n + 1 < N ? n + 1 : n)]"),
    "nf4 codes 12 and 13 swapped": (
        "tg_oracle.c",
        "    0.44070982933044434,\n    0.5626170039176941,",
        "    0.5626170039176941,\n    0.44070982933044434,"),
    "nf4 code 3 mistyped": (
        "tg_oracle.c",
        "-0.39491748809814453,",
        "-0.39591748809814453,"),
    "nf4 code used at full precision in the product": (
        "tg_oracle.c",
        "tg_oracle_f16_to_f64(tg_oracle_f64_to_f16(kNf4Codes[nib]))",
        "kNf4Codes[nib]"),
    "nf4 nibble order reversed": (
        "tg_oracle.c",
        "(word >> (4u * (uint32_t)(n % 8))) & 15u",
        "(word >> (4u * (uint32_t)(7 - n % 8))) & 15u"),
    "nf4 scale group of half the rows": (
        "tg_oracle.c",
        "const int64_t g = k / group; /* scale row */",
        "const int64_t g = k / (group > 1 ? group / 2 : 1);"),
    "GELU-tanh cubic coefficient 0.05": (
        "tg_oracle.c",
        "0.044715 * x * x * x",
        "0.05 * x * x * x"),
    "GELU-tanh sqrt(pi/2) for sqrt(2/pi)": (
        "tg_oracle.c",
        "sqrt(2.0 / acos(-1.0))",
        "sqrt(acos(-1.0) / 2.0)"),
    "GELU erf(x/2) for erf(x/sqrt 2)": (
        "tg_oracle.c",
        "erf(x / sqrt(2.0))",
        "erf(x / 2.0)"),
    "relu backward masks on dC instead of C": (
        "__init__.py",
        "pos = C > np.float16(0)",
        "pos = dC > np.float16(0)"),
    "relu backward passes C == 0": (
        "__init__.py",
        "pos = C > np.float16(0)",
        "pos = C >= np.float16(0)"),
    "dA = dZ B instead of dZ B^T": (
        "__init__.py",
        "dA = gemm_relu(dZ, np.ascontiguousarray(np.asarray(B, np.float16).T), relu=False)",
        "dA = gemm_relu(dZ, np.ascontiguousarray(np.asarray(B, np.float16)), relu=False)"),
}


def _copy_and_run_pins(tmp_path, fname=None, old=None, new=None):
    for d in ("tests", "oracle", "fp16_gemm_relu_gb300"):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "lib"))
    if fname is not None:
        path = tmp_path / "oracle" / fname
        src = path.read_text()
        assert src.count(old) == 1, f"mutation site not unique in {fname}: {old!r}"
        path.write_text(src.replace(old, new))
    return subprocess.run([sys.executable, "-m", "pytest", *PIN_TESTS, "-q", "-x",
                           "-m", "not gpu and not slow", "-p", "no:cacheprovider"],
                          cwd=tmp_path, capture_output=True, text=True, timeout=600)


@pytest.mark.slow
def test_unmutated_copy_passes(tmp_path):
    # the control: the copied tree itself is sound, so a failure below comes from the mistake
    run = _copy_and_run_pins(tmp_path)
    assert run.returncode == 0, run.stdout[-800:]


@pytest.mark.slow
@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    run = _copy_and_run_pins(tmp_path, *MUTANTS[name])
    assert run.returncode != 0, f"no pin failed with the planted mistake: {name}\n{run.stdout[-600:]}"
    assert "failed" in run.stdout, run.stdout[-600:]
