"""Planted mistakes in the oracle: each one must fail at least one pin.

Every case copies the oracle's C source, makes one plausible mistake in the
copy and builds it with the oracle's own flags. The mistakes are a dropped
term, a wrong sign, index, bias or rounding rule, a transposed operand, or
another accumulation order. The case then runs the oracle pin tests against
that build in a child process. The pins must pass on the unchanged source
(the control case) and fail on every mutant. A mutant that survives is a
mistake that no pin would notice.

The mistakes go into copies under ``oracle/_build/mutants/``, on the CPU. The
oracle's own source is never edited, and nothing here touches the GPU library.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qmv_oracle.c")
WORK = os.path.join(ROOT, "oracle", "_build", "mutants")

PIN_FILES = {
    "fp16": "tests/test_oracle_fp16.py",
    "pack": "tests/test_oracle_pack.py",
    "gemv": "tests/test_oracle_gemv.py",
    "norm": "tests/test_oracle_rmsnorm.py",
    "argmax": "tests/test_oracle_argmax.py",
}

# (name, area whose pins run first, [(old text, new text, occurrence)]).
# occurrence None: the old text must occur exactly once; n: replace the n-th.
MUTANTS = [
    # binary16 <-> binary32
    ("f16_exponent_bias", "fp16", [("(e - 15u + 127u) << 23", "(e - 14u + 127u) << 23", None)]),
    ("f16_subnormal_scale", "fp16", [("(1.0f / 16777216.0f)", "(1.0f / 8388608.0f)", None)]),
    ("f16_subnormal_sign_lost", "fp16", [("return sign ? -v : v;", "return v;", None)]),
    ("f32_to_f16_ties_away", "fp16", [("(rem == 0x1000u && (hv & 1u))", "(rem == 0x1000u)", None)]),
    ("f32_to_f16_round_threshold", "fp16", [("rem > 0x1000u ||", "rem > 0x1001u ||", None)]),
    ("f32_to_f16_overflow_edge", "fp16", [("if (e > 15)", "if (e > 16)", None)]),
    ("f32_to_f16_normal_edge", "fp16", [("if (e >= -14)", "if (e >= -15)", None)]),
    ("f32_to_f16_subnormal_shift", "fp16", [("int shift = -e - 1;", "int shift = -e - 2;", None)]),
    ("f16_nan_payload_dropped", "fp16", [("sign | 0x7F800000u | (m << 13)", "sign | 0x7F800000u", None)]),
    ("f32_to_f16_nan_to_inf", "fp16", [("(uint16_t)(sign | 0x7E00u | ((ax >> 13) & 0x3FFu))",
                                        "(uint16_t)(sign | 0x7C00u)", None)]),
    ("f32_to_f16_inf_sign_lost", "fp16", [("return (uint16_t)(sign | 0x7C00u);\n", "return (uint16_t)(0x7C00u);\n", 0)]),
    ("f32_to_f16_carry_lost", "fp16", [("            hv += 1;                     /* a carry",
                                        "            hv = (hv & ~0x3FFu) | ((hv + 1) & 0x3FFu);  /* a carry", None)]),
    ("f32_to_f16_underflow_sign_lost", "fp16", [("return sign;                     /* below half",
                                                 "return 0;                        /* below half", None)]),
    # packer and decoder
    ("pack_twos_complement", "pack", [("int u = v + bias;", "int u = v;", None)]),
    ("pack_msb_first", "pack", [("<< (bits * (int)(k % per_word))",
                                 "<< (bits * (int)(per_word - 1 - k % per_word))", None)]),
    ("unpack_msb_first", "pack", [("(w >> (bits * (int)(k % per_word)))",
                                   "(w >> (bits * (int)(per_word - 1 - k % per_word)))", None)]),
    ("unpack_offset_dropped", "pack", [("(int8_t)((int)u - bias)", "(int8_t)((int)u)", None)]),
    ("pack_range_off_by_one", "pack", [("v >= bias", "v > bias", None)]),
    ("pack_word_index", "pack", [("words[n * wpr + k / per_word] |=",
                                  "words[n * wpr + k % wpr] |=", None)]),
    ("unpack_mask_wide", "pack", [("(w >> (bits * (int)(k % per_word))) & mask;",
                                   "(w >> (bits * (int)(k % per_word))) & (mask | (mask << 1));", None)]),
    # residual add + RMSNorm
    ("residual_sign", "norm", [("orc_f16_to_f32(x[k]) + orc_f16_to_f32(r[k])",
                                "orc_f16_to_f32(x[k]) - orc_f16_to_f32(r[k])", None)]),
    ("fused_residual_sign", "norm", [("orc_f16_to_f32(xm[k]) + orc_f16_to_f32(rm[k])",
                                      "orc_f16_to_f32(xm[k]) - orc_f16_to_f32(rm[k])", 0)]),
    ("fused_norms_x_not_h", "norm", [("float hv = orc_f16_to_f32(orc_f32_to_f16(s));",
                                      "float hv = orc_f16_to_f32(xm[k]);", None)]),
    ("fused_squares_unrounded_h", "norm", [("float hv = orc_f16_to_f32(hk);", "float hv = s;", None)]),
    ("sumsq_term_dropped", "norm", [("blk = blk + sq;", "blk = sq;", 0)]),
    ("fused_sumsq_term_dropped", "norm", [("blk = blk + sq;", "blk = sq;", 1)]),
    ("sumsq_blocks_not_added", "norm", [("ss = ss + blk;", "ss = blk;", 0)]),
    ("norm_serial_sum_of_squares", "norm", [("float inv = orc_rms_inv(orc_sumsq(h, K, order), K, eps);",
                                             "float inv = orc_rms_inv(orc_sumsq(h, K, 1), K, eps);", None),
                                            ("blk = blk + sq;", "ss = ss + sq;", 1)]),
    ("fused_ragged_block_lost", "norm", [("if ((k + 1) % ORC_BLOCK == 0 || k + 1 == K) {",
                                          "if ((k + 1) % ORC_BLOCK == 0) {", None)]),
    ("rms_eps_dropped", "norm", [("float t = mean + eps;", "float t = mean;", None)]),
    ("rms_mean_over_k_minus_1", "norm", [("float mean = ss / (float)K;",
                                          "float mean = ss / (float)(K - 1);", None)]),
    ("inv_in_double", "norm", [("float inv = 1.0f / rt;", "float inv = (float)(1.0 / sqrt((double)t));", None),
                               ("inv = 1.0f / rt;", "inv = (float)(1.0 / sqrt((double)t));", 0)]),
    ("mean_by_reciprocal", "norm", [("float mean = ss / (float)K;", "float mean = ss * (1.0f / (float)K);", None),
                                    ("mean = ss / (float)K;", "mean = ss * (1.0f / (float)K);", 0)]),
    ("fused_sqrt_dropped", "norm", [("inv = 1.0f / rt;", "inv = 1.0f / t;", 1)]),
    ("rmsnorm_gamma_dropped", "norm", [("float b = a * orc_f16_to_f32(gamma[k]);", "float b = a;", 0)]),
    ("fused_gamma_dropped", "norm", [("float b = a * orc_f16_to_f32(gamma[k]);", "float b = a;", 1)]),
    ("rmsnorm_one_plus_gamma", "norm", [("float b = a * orc_f16_to_f32(gamma[k]);",
                                         "float b = a * (1.0f + orc_f16_to_f32(gamma[k]));", 0)]),
    ("norm_scale_before_normalise", "norm", [
        ("float a = orc_f16_to_f32(h[k]) * inv;", "float a = orc_f16_to_f32(h[k]) * orc_f16_to_f32(gamma[k]);", None),
        ("float b = a * orc_f16_to_f32(gamma[k]);", "float b = a * inv;", 0),
        ("float a = hv * inv;", "float a = hv * orc_f16_to_f32(gamma[k]);", None),
        ("float b = a * orc_f16_to_f32(gamma[k]);", "float b = a * inv;", 0)]),
    # matvec
    ("gemv_block_term_dropped", "gemv", [("p = p + prod;", "p = prod;", None)]),
    ("gemv_blocks_not_added", "gemv", [("if (b0 == g0) q = p; else q = q + p;", "q = p;", None)]),
    ("gemv_groups_not_added", "gemv", [("acc = acc + t;", "acc = t;", None)]),
    ("gemv_scale_transposed", "gemv", [("scales[n * G + g]", "scales[g * N + n]", None)]),
    ("gemv_first_scale_only", "gemv", [("scales[n * G + g]", "scales[n * G]", None)]),
    ("gemv_codes_reversed_in_block", "gemv", [("(float)vn[k]", "(float)vn[b1 - 1 - (k - b0)]", None)]),
    ("gemv_wrong_column", "gemv", [("const uint16_t *ym = y + m * K;", "const uint16_t *ym = y;", None)]),
    ("gemv_scale_step_fused", "gemv", [("acc = acc + t;",
                                        "acc = fmaf(q, orc_f16_to_f32(scales[n * G + g]), acc); (void)t;",
                                        None)]),
    ("gemv_block_in_double", "gemv", [("float p = 0.0f;", "double p = 0.0;", None)]),
    ("gemv_group_dot_in_double", "gemv", [("float q = 0.0f;", "double q = 0.0;", None)]),
    ("gemv_group_one_chain", "gemv", [("b0 < g1; b0 += ORC_BLOCK)", "b0 < g1; b0 = g1)", None),
                                      ("b0 + ORC_BLOCK < g1 ? b0 + ORC_BLOCK : g1", "g1", None)]),
    ("block_of_16", "gemv", [("#define ORC_BLOCK 32", "#define ORC_BLOCK 16", None)]),
    # argmax
    ("argmax_last_max", "argmax", [("y[n] > y[best]", "y[n] >= y[best]", None)]),
    ("argmax_best_starts_at_0", "argmax", [("int64_t best = -1;", "int64_t best = 0;", None)]),
    ("argmax_value_of_last", "argmax", [("*max_out = y[best];", "*max_out = y[N - 1];", None)]),
    ("argmax_abs_compare", "argmax", [("y[n] > y[best]", "fabsf(y[n]) > fabsf(y[best])", None)]),
    ("argmax_nan_not_skipped", "argmax", [("if (y[n] != y[n]) continue;", "(void)0;", None)]),
]

# Runs in the child: load the oracle package under its own name, point its
# build at the mutant source, then run the pin files with pytest.
_RUNNER = r"""
import importlib.util, os, sys
root, src, build = sys.argv[1:4]
spec = importlib.util.spec_from_file_location("oracle", os.path.join(root, "oracle", "__init__.py"))
mod = importlib.util.module_from_spec(spec)
spec.loader.exec_module(mod)
mod._SRC = src
mod._BUILD_DIR = build
mod._LIB_PATH = os.path.join(build, "liboracle.so")
sys.modules["oracle"] = mod
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider", "-W", "ignore", *sys.argv[4:]]))
"""


def _mutate(text, edits):
    for old, new, occ in edits:
        n = text.count(old)
        if occ is None:
            assert n == 1, f"{old!r} occurs {n} times"
            text = text.replace(old, new)
        else:
            assert n > occ, f"{old!r} occurs {n} times"
            at = -1
            for _ in range(occ + 1):
                at = text.index(old, at + 1)
            text = text[:at] + new + text[at + len(old):]
    return text


def _run(name, area, edits):
    d = os.path.join(WORK, name)
    shutil.rmtree(d, ignore_errors=True)
    os.makedirs(d)
    with open(SRC) as f:
        text = _mutate(f.read(), edits)
    src = os.path.join(d, "qmv_oracle.c")
    with open(src, "w") as f:
        f.write(text)
    # build here, so that a mutant that does not compile is reported as such
    # and not counted as caught; the child then finds the library up to date
    b = subprocess.run(["gcc", *oracle.CFLAGS, "-o", os.path.join(d, "liboracle.so"), src, "-lm"],
                       capture_output=True, text=True)
    if b.returncode != 0:
        return "build failed", b.stderr[-2000:]
    files = [PIN_FILES[area]] + [p for a, p in PIN_FILES.items() if a != area]
    p = subprocess.run([sys.executable, "-c", _RUNNER, ROOT, src, d, *files],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    return p.returncode, (p.stdout + p.stderr)[-2000:]


@pytest.fixture(scope="module")
def outcomes():
    cases = [("control", "gemv", [])] + MUTANTS
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        futs = {c[0]: ex.submit(_run, *c) for c in cases}
        return {k: f.result() for k, f in futs.items()}


def test_mutant_names_unique():
    names = [m[0] for m in MUTANTS]
    assert len(names) == len(set(names))


def test_control_passes(outcomes):
    rc, log = outcomes["control"]
    assert rc == 0, log


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(outcomes, name):
    rc, log = outcomes[name]
    # pytest exit code 1: tests ran and at least one pin failed (not a build
    # or collection error, which would be 2..4, nor a crash)
    assert rc == 1 and " failed" in log, f"mutant {name} survived or broke the run (rc {rc}):\n{log}"
