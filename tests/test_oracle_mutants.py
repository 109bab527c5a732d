"""The oracle's pins have teeth: plant a plausible mistake in a copy of
oracle.c (on the CPU), build it, and check that the pin tests fail on it."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "q4_0 nibble order swapped": ("(uint8_t)(q0 | (q1 << 4))", "(uint8_t)(q1 | (q0 << 4))"),
    "q4_0 d sign dropped": ("const float d = vmax / -8.0f;", "const float d = vmax / 8.0f;"),
    "q4_K min term dropped": ("acc += t1 - t2;", "acc += t1;"),
    "q4_K min sign flipped": ("acc += t1 - t2;", "acc += t1 + t2;"),
    "scale high bits from wrong byte": ("((q[j - 4] >> 6) << 4)", "((q[j] >> 6) << 4)"),
    "q4_K high nibble paired with wrong activations": (
        "hi += (x[b].qs[32 * c + l] >> 4) * y[b].qs[64 * c + 32 + l];",
        "hi += (x[b].qs[32 * c + l] >> 4) * y[b].qs[64 * c + 16 + l];"),
    "q8 rounding truncates": ("return floorf(v + 0.5f);", "return floorf(v);"),
    "bsums sum one element": ("s += y[b].qs[16 * t + i];", "s += y[b].qs[16 * t];"),
    "w4a16 nibble order reversed": ("<< (4 * i);", "<< (4 * (7 - i));"),
    "mul_mat output transposed": ("Y32[m * nrows + r] =", "Y32[r * M + m] ="),
    "fp16 ties away from zero": ("if (rem > half || (rem == half && (q & 1))) q += 1;",
                                 "if (rem >= half) q += 1;"),
    "q6_K ql high nibble from wrong element": (
        "((u[64 * c + 32 + l] & 15) << 4)", "((u[64 * c + 16 + l] & 15) << 4)"),
    "q6_K qh field order reversed": ("(blk->qh[32 * h + (r % 32)] >> (2 * (r / 32))) & 3",
                                     "(blk->qh[32 * h + (r % 32)] >> (6 - 2 * (r / 32))) & 3"),
    "q6_K code offset off by one": ("return (lo | (hi << 4)) - 32;", "return (lo | (hi << 4)) - 31;"),
    "q6_K group index transposed": ("q6_K_code(&x[b], 16 * j + i) * y[b].qs[16 * j + i];",
                                    "q6_K_code(&x[b], 16 * j + i) * y[b].qs[16 * i + j];"),
    "q6_K scale sign dropped": ("sc[j] = vmax / -32.0f;", "sc[j] = fabsf(vmax) / 32.0f;"),
    "q6_K activation scale dropped": ("acc += (y[b].d * orc_fp16_to_fp32(x[b].d)) * (float)isum;",
                                      "acc += orc_fp16_to_fp32(x[b].d) * (float)isum;"),
    "w4a16 lut indexed by the wrong nibble": (
        "wh[kk] = (double)orc_fp16_to_fp32(scales[n * ng + g]) * (double)orc_fp16_to_fp32(lut[q]);",
        "wh[kk] = (double)orc_fp16_to_fp32(scales[n * ng + g]) * (double)orc_fp16_to_fp32(lut[q ^ 1]);"),
    "q4_0 zero point off by one": ("int q0 = clampi((int)floorf(v0 + 8.5f), 0, 15);",
                                   "int q0 = clampi((int)floorf(v0 + 7.5f), 0, 15);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {old}"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
                    "-I", os.path.join(ROOT, "oracle"), "-o", str(so), str(mut), "-lm"], check=True)
    env = dict(os.environ, QMM_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant '{name}'\n{r.stdout[-2000:]}"
