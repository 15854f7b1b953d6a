"""The pins are strong enough: each plants one plausible mistake in a copy of
the oracle's C source (on the CPU, in a temporary directory) and checks that
the oracle pins and the golden fixtures reject that copy.

Every mutant keeps its loops finite and its indices in bounds, so a mutant
can only give wrong numbers, never hang or crash the check.  Each one runs the
pin modules in a child pytest (stopping at the first failure) with the
``orc`` fixture pointed at the mutant build.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "clef_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_golden.py"),
        os.path.join(ROOT, "tests", "test_oracle_pins.py")]

# (name, text in the oracle source, replacement); each text occurs exactly once
MUTANTS = [
    ("rotation: butterfly difference reversed",
     "float a = v[i], b = v[i + h];\n                v[i] = a + b;\n                v[i + h] = a - b;",
     "float a = v[i], b = v[i + h];\n                v[i] = a + b;\n                v[i + h] = b - a;"),
    ("rotation: normalisation dropped",
     "const float c = wht_c();", "const float c = 1.0f;"),
    ("rotation: last butterfly stage skipped",
     "for (int h = 1; h < 128; h <<= 1)\n        for (int i = 0; i < 128; i++)\n"
     "            if ((i & h) == 0) {\n                float a",
     "for (int h = 1; h < 64; h <<= 1)\n        for (int i = 0; i < 128; i++)\n"
     "            if ((i & h) == 0) {\n                float a"),
    ("rotation: every other 128-block left unrotated",
     "for (int64_t b = 0; b < K; b += 128)", "for (int64_t b = 0; b < K; b += 256)"),
    ("int8: scale divisor 128",
     "*s = amax / 127.0f;\n    const float r = 127.0f / amax;",
     "*s = amax / 128.0f;\n    const float r = 128.0f / amax;"),
    ("int8: codes truncated instead of rounded",
     "float t = rne_int(v[k] * r);", "float t = truncf(v[k] * r);"),
    ("int8: ties rounded up instead of to even",
     "return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;", "return fl + 1.0f;"),
    ("gemm: weight row read backwards",
     "a += (int64_t)qx[m * K + k] * (int64_t)qw[n * K + k];",
     "a += (int64_t)qx[m * K + k] * (int64_t)qw[n * K + (K - 1 - k)];"),
    ("epilogue: weight scale dropped",
     "float y = ((float)acc * s_m) * sw_n;", "float y = (float)acc * s_m;"),
    ("epilogue: bias dropped",
     "y = y + bf16_to_f32(bias[n]);", "y = y + 0.0f * bf16_to_f32(bias[n]);"),
    ("swiglu: gate and up swapped",
     "float u = epilogue_f32(acc[N + n], sx[m], sw_gu[N + n], bias_gu, N + n);\n"
     "            h[m * ldh + n] = f32_to_bf16(swiglu_f32(g, u));",
     "float u = epilogue_f32(acc[N + n], sx[m], sw_gu[N + n], bias_gu, N + n);\n"
     "            h[m * ldh + n] = f32_to_bf16(swiglu_f32(u, g));"),
    ("swiglu: sigmoid of -g",
     "float e = expf(-g);", "float e = expf(g);"),
    ("bf16: rounding truncates",
     "if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))\n        keep += 1u;",
     "if (0)\n        keep += 1u;"),
    ("e4m3: ties away from zero",
     "if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0))\n        fl += 1.0;\n    int m = (int)fl;",
     "if (fr >= 0.5)\n        fl += 1.0;\n    int m = (int)fl;"),
    ("e4m3: subnormal spacing 2^-10",
     "double t = ldexp(a, 9), fl", "double t = ldexp(a, 10), fl"),
    ("fp8: scale for a maximum of 240",
     "*s = amax / 448.0f;", "*s = amax / 240.0f;"),
    ("fp8 linear: weight scale dropped",
     "float v = (acc * sx[m]) * sw[n];", "float v = acc * sx[m];"),
    ("lora: base y dropped",
     "y[m * ldy + n] = f32_to_bf16(bf16_to_f32(y[m * ldy + n]) + z);",
     "y[m * ldy + n] = f32_to_bf16(z);"),
    ("lora: B read transposed",
     "double b = (j < r) ? (double)bf16_to_f32(B[n * r + j]) : 0.0;",
     "double b = (j < r) ? (double)bf16_to_f32(B[j * N + n]) : 0.0;"),
    ("fp8 gate/up: gate and up swapped",
     "h[m * ldh + n] = f32_to_bf16(swiglu_f32(gu[0], gu[1]));",
     "h[m * ldh + n] = f32_to_bf16(swiglu_f32(gu[1], gu[0]));"),
    ("unfused swiglu: up read from the gate half",
     "float u = bf16_to_f32(y_gu[m * ldg + N + n]);", "float u = bf16_to_f32(y_gu[m * ldg + n]);"),
    ("fp8: rotation flag ignored",
     "        if (rotate)\n            orc_rotate_rows_f32(x + m * ldx, 1, K, ldx, v);\n        else\n"
     "            for (int64_t k = 0; k < K; k++)\n                v[k] = bf16_to_f32(x[m * ldx + k]);\n"
     "        quant_row_fp8(",
     "        if (0)\n            orc_rotate_rows_f32(x + m * ldx, 1, K, ldx, v);\n        else\n"
     "            for (int64_t k = 0; k < K; k++)\n                v[k] = bf16_to_f32(x[m * ldx + k]);\n"
     "        quant_row_fp8("),
    ("static: scale used as the reciprocal",
     "const float r = 1.0f / s;", "const float r = s;"),
    ("lora: padding columns not zero",
     "t[m * r_pad + j] = 0;", "t[m * r_pad + j] = 0x3F80;"),
    ("fp8 linear: bias dropped",
     "            if (bias)\n                v = v + bf16_to_f32(bias[n]);",
     "            if (bias)\n                v = v + 0.0f * bf16_to_f32(bias[n]);"),
    ("static int8: lower clamp at -128",
     "if (c < -127.0f) c = -127.0f;", "if (c < -128.0f) c = -128.0f;"),
    ("int8: all-zero row gets scale 1",
     "    if (amax == 0.0f) {\n        *s = 0.0f;\n        memset(q, 0, (size_t)K);\n        return;\n    }\n"
     "    *s = amax / 127.0f;",
     "    if (amax == 0.0f) {\n        *s = 1.0f;\n        memset(q, 0, (size_t)K);\n        return;\n    }\n"
     "    *s = amax / 127.0f;"),
    ("int8: absmax over the first 128-block only",
     "    float amax = 0.0f;\n    for (int64_t k = 0; k < K; k++)\n        amax = fmaxf(amax, fabsf(v[k]));\n"
     "    if (amax == 0.0f) {\n        *s = 0.0f;\n        memset(q, 0, (size_t)K);\n        return;\n    }\n"
     "    *s = amax / 127.0f;",
     "    float amax = 0.0f;\n    for (int64_t k = 0; k < 128; k++)\n        amax = fmaxf(amax, fabsf(v[k]));\n"
     "    if (amax == 0.0f) {\n        *s = 0.0f;\n        memset(q, 0, (size_t)K);\n        return;\n    }\n"
     "    *s = amax / 127.0f;"),
    ("lora: t rounded by truncation",
     "t[m * r_pad + j] = f64_to_bf16(a);",
     "{ float tf = (float)a; uint32_t tu; memcpy(&tu, &tf, 4); t[m * r_pad + j] = (uint16_t)(tu >> 16); }"),
]


def _run(tmp, i, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutant '{name}': its text must occur once in the oracle"
    path = os.path.join(tmp, f"mutant_{i}.c")
    with open(path, "w") as f:
        f.write(text.replace(old, new))
    env = dict(os.environ, CLEF_ORACLE_MUTANT=path)
    p = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    return name, p.returncode, p.stdout[-400:]


def test_every_planted_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max(1, min(8, (os.cpu_count() or 2) // 2))) as ex:
        res = list(ex.map(lambda a: _run(str(tmp_path), *a),
                          [(i, *m) for i, m in enumerate(MUTANTS)]))
    missed = [(name, out) for name, rc, out in res if rc == 0]
    assert not missed, "mutants the pins accept: " + "; ".join(n for n, _ in missed)
    # a mutant must be rejected by a failing pin, not by a collection or build error
    for name, rc, out in res:
        assert rc == 1, (name, rc, out)


def test_unmutated_copy_passes(tmp_path):
    """The harness itself: a copy of the unchanged source passes every pin."""
    name, rc, out = _run(str(tmp_path), "none", "none", "#include <math.h>", "#include <math.h>")
    assert rc == 0, out
