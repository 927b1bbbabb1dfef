"""The oracle's pins catch plausible mistakes (CPU only).

Each mutant is a copy of the oracle's C source, in a temporary directory,
with one planted error of the kind a restatement of the pages could contain:
a wrong rounding tie, bias, index, sign or bound.  The oracle's pin tests
run against every mutant and must fail on each; an unmutated copy must pass,
so a failure means the planted error was caught and nothing else.  The
exhaustive 2^32 encoder sweep is left out here (it runs in the ordinary
suite); every mutant must be caught by the faster pins alone.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_recipe.py",
        "tests/test_oracle_gemm.py", "tests/test_oracle_layernorm.py",
        "tests/test_oracle_optimizer.py", "tests/test_oracle_allreduce.py"]

# name: (text in oracle/fp8_oracle.c, replacement); each text occurs once
MUTANTS = {
    "FP8 ties go to the odd code": (
        "code = (lo % 2 == 0) ? lo : hi;           /* tie: even code */",
        "code = (lo % 2 == 1) ? lo : hi;"),
    "E4M3 exponent bias 8 instead of 7": (
        "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    "E5M2 subnormal step 2^-15 instead of 2^-16": (
        "v = ldexp((double)m, -16);", "v = ldexp((double)m, -15);"),
    "encode drops the sign": (
        "return (uint8_t)((neg << 7) | code);", "return (uint8_t)code;"),
    "transposed copy written untransposed": (
        "out_t[c * rows + r] = q;", "out_t[r * cols + c] = q;"),
    "scale multiplied by 2^margin instead of 2^-margin": (
        "float s = (float)ldexp((double)q, -margin);   /* exact, then one rounding */",
        "float s = (float)ldexp((double)q, margin);"),
    "history not shifted before the push": (
        "hist[i] = hist[i - 1];", "hist[i] = hist[i];"),
    "no FLT_MAX clamp of an overflowing scale": (
        "            s = FLT_MAX;\n        *scale = s;", "            s = s;\n        *scale = s;"),
    "amax skips the last element": (
        "for (int64_t i = 0; i < n; ++i) {\n        float a = fabsf(or_bf16_to_f32(x[i]));",
        "for (int64_t i = 0; i < n - 1; ++i) {\n        float a = fabsf(or_bf16_to_f32(x[i]));"),
    "amax lets NaN through": (
        "        float a = fabsf(or_bf16_to_f32(x[i]));\n        if (a > m)",
        "        float a = fabsf(or_bf16_to_f32(x[i]));\n        if (!(a <= m))"),
    "BF16 rounding ties away from zero": (
        "if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))", "if (drop >= 0x8000u)"),
    "GEMM reads B transposed (double path)": (
        "const uint8_t *b = B + j * K;", "const uint8_t *b = B + (N - 1 - j) * K;"),
    "GEMM reads B transposed (exact path)": (
        "y = ib[B[j * K + k]];", "y = ib[B[k * N + j]];"),
    "epilogue drops the second scale": (
        "float sab = sa_inv * sb_inv;", "float sab = sa_inv;"),
    "scale_inv not recomputed": (
        "*scale_inv = 1.0f / s;", "*scale_inv = 1.0f;"),
    # LayerNorm, the FP16 codec, Adam and the FP8 sum
    "LayerNorm variance divided by C - 1": (
        "v /= (double)cols;", "v /= (double)(cols - 1);"),
    "LayerNorm eps added outside the square root": (
        "double rs = 1.0 / sqrt(v + eps);", "double rs = 1.0 / (sqrt(v) + eps);"),
    "LayerNorm beta and gamma swapped": (
        "(double)or_bf16_to_f32(gamma[c]) + (double)or_bf16_to_f32(beta[c]);",
        "(double)or_bf16_to_f32(beta[c]) + (double)or_bf16_to_f32(gamma[c]);"),
    "FP16 ties go to the odd code": (
        "            code = (lo % 2 == 0) ? lo : hi;\n    }\n    return (uint16_t)",
        "            code = (lo % 2 == 1) ? lo : hi;\n    }\n    return (uint16_t)"),
    "FP16 subnormal step 2^-23 instead of 2^-24": (
        "ldexp((double)m, -24)", "ldexp((double)m, -23)"),
    "Adam second moment without the squared gradient": (
        "v = b2 * v + (1.0f - b2) * (g * g);", "v = b2 * v + (1.0f - b2) * g;"),
    "Adam without the first bias correction": (
        "float u = (m / bc1) / (sqrtf(v / bc2) + eps);",
        "float u = m / (sqrtf(v / bc2) + eps);"),
    "Adam weight decay with the wrong sign": (
        "w = w - lr * (u + wd * w);", "w = w - lr * (u - wd * w);"),
    "Adam initial master weights stored unscaled": (
        "w16[i] = or_f16_encode(or_bf16_to_f32(w[i]) * s); /* binary32 multiply */",
        "w16[i] = or_f16_encode(or_bf16_to_f32(w[i]));"),
    "Adam initial weight scale ignores the margin": (
        "        s = (float)ldexp((double)q, -margin);         /* exact, then one rounding */",
        "        s = q;"),
    "FP8 sum multiplied by the scale instead of its inverse": (
        "const float sinv = 1.0f / scale;                   /* binary32 divide */",
        "const float sinv = scale;"),
    "FP8 sum drops the last rank": (
        "for (int32_t r = 0; r < nranks; ++r) {\n            double v = or_fp8_decode",
        "for (int32_t r = 0; r + 1 < nranks; ++r) {\n            double v = or_fp8_decode"),
    "FP8 sum rounds ties away from zero": (
        "if (rest > half || (rest == half && (M & 1)))", "if (rest >= half)"),
    "FP8 sum rounded to binary32 before BF16": (
        "out[i] = bf16_of_exact(acc != 0 && sig != 0 ? neg : 0, P, g + se - 24);\n            continue;",
        "res = (float)((double)acc * ldexp(1.0, g) * (double)sinv);"),
    "FP8 sum without BF16 subnormals": (
        "        u = -133;                                      /* the subnormal quantum 2^-133 */",
        "        u = -126;"),
}


def _run(name, edit):
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        skip = shutil.ignore_patterns("*.so", "*.tmp", "__pycache__", ".pytest_cache")
        shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(tmp, "oracle"), ignore=skip)
        shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(tmp, "tests"), ignore=skip)
        shutil.copy(os.path.join(ROOT, "fp8_workloads.py"), tmp)
        if edit is not None:
            src = os.path.join(tmp, "oracle", "fp8_oracle.c")
            text = open(src).read()
            old, new = edit
            assert text.count(old) == 1, f"{name}: the text to mutate occurs {text.count(old)} times"
            with open(src, "w") as fh:
                fh.write(text.replace(old, new))
        env = dict(os.environ, OMP_NUM_THREADS="2")
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            "-m", "not gpu", "-k", "not exhaustive", *PINS],
                           cwd=tmp, env=env, capture_output=True, text=True, timeout=900)
        return name, r.returncode, (r.stdout + r.stderr)[-1500:]
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_every_planted_mistake_is_caught():
    jobs = [("unmutated control", None)] + list(MUTANTS.items())
    with ThreadPoolExecutor(max_workers=4) as ex:
        results = list(ex.map(lambda job: _run(*job), jobs))
    control = results[0]
    assert control[1] == 0, f"the unmutated copy must pass its pins:\n{control[2]}"
    survivors = [name for name, rc, _ in results[1:] if rc == 0]
    assert not survivors, f"planted mistakes no pin caught: {survivors}"
    # exit status 1 = tests ran and failed; anything else is a broken run
    broken = [(name, rc, out) for name, rc, out in results[1:] if rc != 1]
    assert not broken, broken
