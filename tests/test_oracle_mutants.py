"""The oracle's pins catch plausible mistakes (CPU only).

Each case below plants one mistake in a copy of oracle/qgemm_oracle.c (a
swapped nibble, a dropped sign extension, a wrong index, divisor, clamp,
rounding mode, a dropped or misplaced term), builds it with the oracle's own
flags and runs tests/test_oracle.py against that build in a fresh process.
The run must fail: otherwise the pins would not tell that mistake from the
correct oracle.  The unmodified source, built the same way, must pass.
Every planted mistake stays in bounds, so a mutant fails on its values and
never by reading outside its buffers.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qgemm_oracle.c")

MUTANTS = {
    "s4 unpack reads the nibbles the other way round":
        ("unsigned n = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);",
         "unsigned n = (k % 2 == 0) ? (byte >> 4) : (byte & 0xFu);"),
    "s4 pack swaps the nibbles":
        ("(uint8_t)(((unsigned)lo & 0xFu) | (((unsigned)hi & 0xFu) << 4));",
         "(uint8_t)(((unsigned)hi & 0xFu) | (((unsigned)lo & 0xFu) << 4));"),
    "nibble not sign-extended":
        ("return n < 8u ? (int)n : (int)n - 16;", "return (int)n;"),
    "INT8 GEMM reads B along the wrong k":
        ("acc += (int64_t)A[i * lda + k] * (int64_t)B[j * ldb + k];",
         "acc += (int64_t)A[i * lda + k] * (int64_t)B[j * ldb + (K - 1 - k)];"),
    "int32 overflow not detected":
        ("            if (acc < INT32_MIN || acc > INT32_MAX)\n                return 3;\n", ""),
    "FP16 GEMM reads B along the wrong k":
        ("orc_half_to_double(B[j * ldb + k]);", "orc_half_to_double(B[j * ldb + (K - 1 - k)]);"),
    "W4A16 reads the nibbles the other way round":
        ("int q = nibble_value((k % 2 == 0) ? byte : (unsigned)byte >> 4);",
         "int q = nibble_value((k % 2 == 0) ? (unsigned)byte >> 4 : byte);"),
    "W4A16 uses the next group's scale":
        ("orc_half_to_double(S[n * lds + k / group]);",
         "orc_half_to_double(S[n * lds + (k / group + 1) % (K / group)]);"),
    "quantizer divides the absmax by 8":
        ("orc_float_to_half(a / 7.0f);", "orc_float_to_half(a / 8.0f);"),
    "quantizer clamps at +8":
        ("if (r > 7.0f) r = 7.0f;", "if (r > 8.0f) r = 8.0f;"),
    "quantizer clamps at -7":
        ("if (r < -8.0f) r = -8.0f;", "if (r < -7.0f) r = -7.0f;"),
    "quantizer rounds half away from zero":
        ("float r = rintf(x[t + u] / s);", "float r = roundf(x[t + u] / s);"),
    "low-rank projection reads U in the wrong column":
        ("orc_half_to_double(U[k * ldu + r]);", "orc_half_to_double(U[k * ldu + (R - 1 - r)]);"),
    "W4A4 uses block 0's row scale for every block":
        ("orc_half_to_double(SX[m * ldsx + j])", "orc_half_to_double(SX[m * ldsx + 0])"),
    "W4A4 drops the column scale":
        ("orc_half_to_double(SW[n * ldsw + j]) * (double)dot;", "(double)dot;"),
    "W4A4 reads V in the wrong row":
        ("XU[m * ldxu + r] * orc_half_to_double(V[r * ldv + n]);",
         "XU[m * ldxu + r] * orc_half_to_double(V[(R - 1 - r) * ldv + n]);"),
    "W4A4 drops the bias":
        ("acc += orc_half_to_double(bias[n]);", "acc += 0.0;"),
    "W4A4 column multiplier also scales the bias":
        ("            if (alpha)\n                acc *= orc_half_to_double(alpha[n]);\n"
         "            if (bias)\n                acc += orc_half_to_double(bias[n]);\n",
         "            if (bias)\n                acc += orc_half_to_double(bias[n]);\n"
         "            if (alpha)\n                acc *= orc_half_to_double(alpha[n]);\n"),
}


def _build(source: str, out_dir: str, name: str) -> str:
    src = os.path.join(out_dir, name + ".c")
    lib = os.path.join(out_dir, name + ".so")
    with open(src, "w") as f:
        f.write(source)
    subprocess.run(["gcc"] + oracle.CFLAGS + [src, "-o", lib, "-lm"], check=True)
    return lib


def _pins_pass(lib: str) -> bool:
    env = dict(os.environ, ORACLE_LIB_PATH=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                        "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode == 0


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_source_passes(source, tmp_path):
    assert _pins_pass(_build(source, str(tmp_path), "control"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(source, tmp_path, name):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site not found exactly once: {name}"
    lib = _build(source.replace(old, new), str(tmp_path), "mutant")
    assert not _pins_pass(lib), f"the pins do not catch: {name}"
