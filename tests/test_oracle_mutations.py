"""Planted mistakes in the oracle: every one must fail at least one oracle pin.

Each case copies ``oracle/`` and the oracle pin modules into a temporary
directory, edits one spot of the copied ``qmm_oracle.c`` into a plausible
mistake (another rounding rule, an off-by-one divisor, a swapped bit or nibble
position, a wrong index, a dropped saturation or sign), and runs the pins that
cover that spot against the copy in a child pytest.  The real oracle is never
touched.  A mutant that passes its pins would mean a pin is missing; the
unedited copy must pass them (so a broken harness cannot make every mutant
look caught).
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = "ggml_block_quantized_linear_b300"

FP16 = ["test_oracle_fp16.py"]
Q8 = ["test_oracle_q8_0.py", "test_oracle_ties.py"]
Q4 = ["test_oracle_q4_k.py", "test_oracle_ties.py"]
Q6 = ["test_oracle_q6_k.py", "test_oracle_ties.py"]
KQ = ["test_oracle_kquants.py"]
F8 = ["test_oracle_fp8.py"]
MM = ["test_oracle_matmul.py"]

# name: (text in qmm_oracle.c, replacement, pin modules)
MUTANTS = {
    # binary16 encoder: truncation, or ties away from zero instead of to even
    "f16_truncate": ("double N = rint(ldexp(a, 10 - e));", "double N = floor(ldexp(a, 10 - e));", FP16),
    "f16_ties_away": ("double N = rint(ldexp(a, 10 - e));", "double N = round(ldexp(a, 10 - e));", FP16),
    # Q8_0: divisor, rounding rule, unrounded scale used for the codes
    "q8_div128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;", Q8),
    "q8_rint": ("q = clampf(roundf(x[i] / df), -127.0f, 127.0f);",
                "q = clampf(rintf(x[i] / df), -127.0f, 127.0f);", Q8),
    "q8_unrounded_scale": ("q = clampf(roundf(x[i] / df), -127.0f, 127.0f);",
                           "q = clampf(roundf(x[i] / d), -127.0f, 127.0f);", Q8),
    # Q4_K: sub-block range divisor, rounding, nibble order, scale packing, sign of the min
    "q4_div16": ("s[j] = range / 15.0f;", "s[j] = range / 16.0f;", Q4),
    "q4_rint": ("v = clampf(roundf(shifted / S), 0.0f, 15.0f);",
                "v = clampf(rintf(shifted / S), 0.0f, 15.0f);", Q4),
    "q4_nibbles": ("qs[32 * c + l] = (uint8_t)(q[32 * (2 * c) + l] | (q[32 * (2 * c + 1) + l] << 4));",
                   "qs[32 * c + l] = (uint8_t)(q[32 * (2 * c + 1) + l] | (q[32 * (2 * c) + l] << 4));", Q4),
    "q4_pack_swap": ("s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((mc[j + 4] & 15) << 4));",
                     "s[j + 8] = (uint8_t)((mc[j + 4] & 15) | ((sc[j + 4] & 15) << 4));", Q4),
    "q4_min_sign": ("(qs[32 * c + l] & 15);\n            float prod = S * (float)q;\n            y[32 * j + l] = prod - Mn;",
                    "(qs[32 * c + l] & 15);\n            float prod = S * (float)q;\n            y[32 * j + l] = prod + Mn;",
                    Q4),
    # Q6_K: divisor, rounding, high-bit position
    "q6_div32": ("s[j] = amax / 31.0f;", "s[j] = amax / 32.0f;", Q6),
    "q6_rint": ("int c = S > 0.0f ? (int)clampf(roundf(x[w] / S), -32.0f, 31.0f) : 0;",
                "int c = S > 0.0f ? (int)clampf(rintf(x[w] / S), -32.0f, 31.0f) : 0;", Q6),
    "q6_hibits": ("out[hi_byte] |= (uint8_t)((q >> 4) << hi_shift);",
                  "out[hi_byte] |= (uint8_t)((q >> 4) << (6 - hi_shift));", Q6),
    # Q5_K / Q3_K / Q2_K
    "q5_div32": ("affine_stats(x, 8, 32, 31.0f", "affine_stats(x, 8, 32, 32.0f", KQ),
    "q5_rint": ("q = (int)clampf(roundf((x[32 * j + l] + Mn) / S), 0.0f, 31.0f);",
                "q = (int)clampf(rintf((x[32 * j + l] + Mn) / S), 0.0f, 31.0f);", KQ),
    "q5_qh_order": ("out[16 + l] |= (uint8_t)((q >> 4) << j);", "out[16 + l] |= (uint8_t)((q >> 4) << (7 - j));", KQ),
    "q3_div4": ("s[j] = amax / 3.0f;", "s[j] = amax / 4.0f;", KQ),
    "q3_field": ("sb[8 + j % 4] |= (uint8_t)(((v >> 4) & 3) << (2 * (j / 4)));",
                 "sb[8 + j / 4] |= (uint8_t)(((v >> 4) & 3) << (2 * (j % 4)));", KQ),
    "q3_rint": ("int c = S > 0.0f ? (int)clampf(roundf(x[w] / S), -4.0f, 3.0f) : 0;",
                "int c = S > 0.0f ? (int)clampf(rintf(x[w] / S), -4.0f, 3.0f) : 0;", KQ),
    "q2_nibbles": ("out[j] = (uint8_t)(sc | (mc << 4));", "out[j] = (uint8_t)(mc | (sc << 4));", KQ),
    "q2_div16": ("uint16_t d16 = orc_f32_to_f16(smax / 15.0f);\n    uint16_t dmin16 = orc_f32_to_f16(mmax / 15.0f);",
                 "uint16_t d16 = orc_f32_to_f16(smax / 16.0f);\n    uint16_t dmin16 = orc_f32_to_f16(mmax / 15.0f);", KQ),
    "q2_rint": ("q = (int)clampf(roundf((x[w] + Mn) / S), 0.0f, 3.0f);",
                "q = (int)clampf(rintf((x[w] + Mn) / S), 0.0f, 3.0f);", KQ),
    # FP8 E4M3: row-scale divisor, ties away, no saturation
    "fp8_div447": ("float s = amax / 448.0f;", "float s = amax / 447.0f;", F8),
    "fp8_ties_away": ("double v = ldexp(rint(ldexp(a, 3 - e)), e - 3);",
                      "double v = ldexp(round(ldexp(a, 3 - e)), e - 3);", F8),
    "fp8_no_saturation": ("    if (v > 448.0)\n        v = 448.0;\n", "", F8),
    # matmul: reversed activation index (a transposed / misaligned operand), fp32 accumulation
    "mm_reversed_k": ("double p = (double)w[k] * (double)orc_bf16_to_f32(xm[k]);",
                      "double p = (double)w[k] * (double)orc_bf16_to_f32(xm[K - 1 - k]);", MM),
    "mm_f32_accumulation": ("double acc = 0.0, aacc = 0.0;", "float acc = 0.0f; double aacc = 0.0;", MM),
}


def run_pins(edit, modules):
    """Copy the oracle and the pins, apply `edit` (None: no edit), run the pins;
    returns (pytest exit code, last output line)."""
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(tmp, "oracle"),
                        ignore=shutil.ignore_patterns("_build", "__pycache__"))
        os.makedirs(os.path.join(tmp, "tests"))
        for name in set(modules) | {"conftest.py", "test_oracle_q4_k.py"}:
            shutil.copy(os.path.join(ROOT, "tests", name), os.path.join(tmp, "tests", name))
        shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tmp, "tests", "golden"))
        os.symlink(os.path.join(ROOT, PKG), os.path.join(tmp, PKG))
        if edit is not None:
            path = os.path.join(tmp, "oracle", "qmm_oracle.c")
            src = open(path).read()
            assert src.count(edit[0]) == 1, "mutation site not unique or missing: %r" % edit[0][:60]
            open(path, "w").write(src.replace(edit[0], edit[1]))
        env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONDONTWRITEBYTECODE="1")
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            "-m", "not gpu"] + ["tests/" + m for m in modules],
                           cwd=tmp, env=env, capture_output=True, text=True, timeout=600)
        lines = (r.stdout.strip() or r.stderr.strip()).splitlines()
        return r.returncode, lines[-1] if lines else ""
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_every_planted_mistake_fails_a_pin():
    jobs = {"(unedited)": (None, sorted({m for *_, ms in MUTANTS.values() for m in ms}))}
    jobs.update({name: ((old, new), ms) for name, (old, new, ms) in MUTANTS.items()})
    with concurrent.futures.ThreadPoolExecutor(max(1, min(8, (os.cpu_count() or 2) // 2))) as ex:
        res = dict(zip(jobs, ex.map(lambda j: run_pins(*j), jobs.values())))
    rc, last = res.pop("(unedited)")
    assert rc == 0, "the unedited oracle copy fails its pins: " + last
    survivors = {name: last for name, (rc, last) in res.items() if rc != 1}
    assert not survivors, "planted mistakes not caught by any pin: %s" % survivors
