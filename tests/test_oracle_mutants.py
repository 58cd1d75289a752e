"""Mutation check of the oracle's pins (CPU only).

Each mutant is a copy of the oracle's C source with one plausible mistake
planted (a dropped term, a wrong sign, index or operand order, a wrong
constant, a wrong reading of the layout); it is compiled into a temporary
directory and the pin battery runs against it in a child process.  Every
mutant must fail at least one pin other than the golden digest, which is a
regression check and not an independent pin (a mutant that crashes the
child counts as caught).  The oracle itself is never
modified.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# Mutant builds live inside the repository tree (git-ignored).
_SCRATCH = os.path.join(ROOT, "tests", "_mutants")

# (name, [(old, new), ...]); every `old` must occur exactly once in the source.
MUTANTS = [
    ("chunk drops its last square", [("for (int k = 1; k < 8; ++k)", "for (int k = 1; k < 7; ++k)")]),
    ("tree drops its last level", [("for (int o = P / 2; o >= 1; o /= 2)", "for (int o = P / 2; o > 1; o /= 2)")]),
    ("chunks of 4 instead of 8", [("int C = D / 8;", "int C = D / 4;"),
                                  ("const float* xc = x + 8 * c;", "const float* xc = x + 4 * c;"),
                                  ("for (int k = 1; k < 8; ++k)", "for (int k = 1; k < 4; ++k)")]),
    ("mean over D-1", [("float ms = ss / (float)D;", "float ms = ss / (float)(D - 1);")]),
    ("eps outside the root", [("float t = ms + eps;", "float t = ms;"),
                              ("return 1.0f / rt;", "return 1.0f / (rt + eps);")]),
    ("one rounding for 1/sqrt", [("return 1.0f / rt;", "return (float)(1.0 / sqrt((double)t));")]),
    ("weight index", [("y[d] = xn * w[d];", "y[d] = xn * w[0];")]),
    ("weight before the norm", [("float xn = x[d] * inv;\n        y[d] = xn * w[d];",
                                 "float xn = x[d] * w[d];\n        y[d] = xn * inv;")]),
    ("K normalised with the Q weight", [("const float* w = part == 0 ? wq : wk;",
                                         "const float* w = part == 0 ? wq : wq;")]),
    ("rotation sign", [("*u_out = uc - vs;", "*u_out = uc + vs;")]),
    ("rotation operand", [("float us = u * s;", "float us = v * s;")]),
    ("half-split pairs", [("h3o_rotate_pair(pb->in_dtype, cs[i], sn[i], n[2 * i], n[2 * i + 1],\n"
                           "                        &dst[2 * i], &dst[2 * i + 1]);",
                           "h3o_rotate_pair(pb->in_dtype, cs[i], sn[i], n[i], n[i + R / 2],\n"
                           "                        &dst[i], &dst[i + R / 2]);")]),
    ("every axis uses the t position", [("float p = (float)tok_pos[a];", "float p = (float)tok_pos[0];")]),
    ("frequency exponent i/d", [("double expo = -(2.0 * (double)i) / (double)d;",
                                 "double expo = -(1.0 * (double)i) / (double)d;")]),
    ("pass-through channels zeroed", [("for (int d = R; d < D; ++d) dst[d] = n[d];",
                                       "for (int d = R; d < D; ++d) dst[d] = 0;")]),
    ("quadrant 1 cosine sign", [("case 1: s = cr; c = -sr; break;", "case 1: s = cr; c = sr; break;")]),
    ("series coefficient", [("H3O_S5 = 0x1.111112p-7f", "H3O_S5 = 0x1.111110p-7f")]),
    ("cosine series one term short", [("pc = fmaf(pc, r2, H3O_C4);", "")]),
    ("V not the identity", [("for (int64_t e = 0; e < HD; ++e) yv[e] = vsrc[e];",
                             "for (int64_t e = 0; e < HD; ++e) yv[e] = vsrc[e ^ 1];")]),
    ("token-major output", [("return ((b * pb->heads + h) * pb->seq + s) * pb->head_dim;",
                             "return ((b * pb->seq + s) * pb->heads + h) * pb->head_dim;")]),
    ("valid prefix over the whole batch", [("    return s < vl;\n}", "    return r < vl;\n}")]),
    ("per-item lengths ignored", [("        vl = pb->valid_lens[b];", "        vl = pb->valid_len;")]),
    ("token-major head and token swapped", [
        ("if (pb->out_layout == 1) return ((b * pb->seq + s) * pb->heads + h) * pb->head_dim;",
         "if (pb->out_layout == 1) return ((b * pb->heads + h) * pb->seq + s) * pb->head_dim;")]),
    ("saturation counts the largest code", [("if (fabsf(z) > 448.0f) counts[t] += 1;",
                                             "if (fabsf(z) >= 448.0f) counts[t] += 1;")]),
    ("amax over padded rows", [("        if (!h3o_row_valid(pb, r)) continue;\n"
                                "        h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, y[0], y[1], y[2]);\n"
                                "        for (int t = 0; t < 3; ++t)\n"
                                "            for (int64_t e = 0; e < HD; ++e) {\n"
                                "                float a = fabsf(h3o_widen(pb->in_dtype, y[t][e]));",
                                "        h3o_row16_with(pb, qkv, wq, wk, pos, inv_freq, r, y[0], y[1], y[2]);\n"
                                "        for (int t = 0; t < 3; ++t)\n"
                                "            for (int64_t e = 0; e < HD; ++e) {\n"
                                "                float a = fabsf(h3o_widen(pb->in_dtype, y[t][e]));")]),
    ("descale inverted", [("s = a / 448.0f;", "s = 448.0f / a;")]),
    ("cast divides by the factor", [("float z = v * inv;", "float z = v / inv;")]),
    ("static factor not inverted", [("i = 1.0f / tab;", "i = tab;")]),
    ("e4m3 saturates late", [("if (a >= 448.0f) return (uint8_t)(sign | 0x7Eu);",
                              "if (a > 480.0f) return (uint8_t)(sign | 0x7Eu);")]),
    ("f16 rounds half up", [("uint32_t m = (uint32_t)rintf(n);", "uint32_t m = (uint32_t)floorf(n + 0.5f);")]),
    ("bf16 subnormal exponent", [("h3o_round_sig(a, 7, -126, &E, &m);", "h3o_round_sig(a, 7, -125, &E, &m);")]),
    ("exp reduction tail sign", [("r = fmaf(-k, H3O_LN2_LO, r);", "r = fmaf(k, H3O_LN2_LO, r);")]),
    ("exp series one term short", [("    p = fmaf(p, r, H3O_E2);\n", "")]),
    ("silu denominator sign", [("float d = 1.0f + e;", "float d = 1.0f - e;")]),
    ("swiglu gate and up swapped", [("float g = h3o_widen(dtype, x[r * row_stride + j]);",
                                     "float g = h3o_widen(dtype, x[r * row_stride + f + j]);")]),
    ("residual fused", [("            float t = b * sc;\n            out[i] = residual[i] + t;",
                         "            out[i] = fmaf(b, sc, residual[i]);")]),
    ("residual scale channel", [("float sc = scale[scale_len == 1 ? 0 : c];", "float sc = scale[0];")]),
    ("sage norm rounded to 16 bits", [("h3o_norm_head_f32(x, w, D, pb->eps, n);",
                                       "h3o_norm_head_f32(x, w, D, pb->eps, n);\n    for (int d = 0; d < D; ++d)"
                                       " n[d] = h3o_widen(pb->in_dtype, h3o_round16(pb->in_dtype, n[d]));")]),
    ("sage K without kv_scale", [("out_k[o + d] = y[d] * kv_scale;", "out_k[o + d] = y[d];")]),
    ("sage kv_scale on Q too", [("h3o_head_f32(pb, row + (int64_t)h * D, wq, cs, sn, out_q + o);",
                                 "h3o_head_f32(pb, row + (int64_t)h * D, wq, cs, sn, out_q + o);\n"
                                 "            for (int d = 0; d < D; ++d) out_q[o + d] *= kv_scale;")]),
    ("sage K with the Q weight", [("h3o_head_f32(pb, row + HD + (int64_t)h * D, wk, cs, sn, y);",
                                   "h3o_head_f32(pb, row + HD + (int64_t)h * D, wq, cs, sn, y);")]),
    ("sage V unscaled", [("float sv = h3o_widen(pb->in_dtype, v[d]) * kv_scale;",
                          "float sv = h3o_widen(pb->in_dtype, v[d]);")]),
    ("sage V through bfloat16", [("out_v[o + d] = h3o_f32_to_f16(sv);",
                                  "out_v[o + d] = h3o_f32_to_f16(h3o_bf16_to_f32(h3o_f32_to_bf16(sv)));")]),
    ("sage half-split pairs", [("h3o_rotate_f32(cs[i], sn[i], n[2 * i], n[2 * i + 1], &dst[2 * i], &dst[2 * i + 1]);",
                                "h3o_rotate_f32(cs[i], sn[i], n[i], n[i + R / 2], &dst[i], &dst[i + R / 2]);")]),
    ("sage pass-through zeroed", [("memcpy(dst + R, n + R, sizeof(float) * (size_t)(D - R));",
                                   "memset(dst + R, 0, sizeof(float) * (size_t)(D - R));")]),
    ("f16 widening bias", [("else v = ldexpf((float)(man | 0x400), ex - 25);",
                            "else v = ldexpf((float)(man | 0x400), ex - 24);")]),
    ("scale accepts subnormals", [("return s >= FLT_MIN && s <= FLT_MAX;", "return s > 0.0f && s <= FLT_MAX;")]),
    ("scale accepts infinity", [("return s >= FLT_MIN && s <= FLT_MAX;", "return s >= FLT_MIN;")]),
    ("smallest normal scale rejected", [("return s >= FLT_MIN && s <= FLT_MAX;",
                                         "return s > FLT_MIN && s <= FLT_MAX;")]),
    ("zero amax gives descale 0", [("i = 448.0f / a;\n            } else {\n                s = 1.0f;",
                                    "i = 448.0f / a;\n            } else {\n                s = 0.0f;")]),
    ("degenerate static entry keeps its factor", [("i = 1.0f / tab;\n            } else {\n                s = 1.0f;\n"
                                                   "                i = 1.0f;",
                                                   "i = 1.0f / tab;\n            } else {\n                s = 1.0f;\n"
                                                   "                i = 1.0f / tab;")]),
    ("amax keeps NaN", [("if (a > m[t]) m[t] = a;", "if (!(a <= m[t])) m[t] = a;")]),
    ("single-tensor amax keeps NaN", [("if (a > m) m = a;", "if (!(a <= m)) m = a;")]),
    ("mean square clamped away from zero", [("float t = ms + eps;", "float t = fmaxf(ms + eps, 1e-30f);")]),
    ("infinite sum clamped", [("float rt = sqrtf(t);", "float rt = sqrtf(fminf(t, FLT_MAX));")]),
]

_CHILD = r"""
import os, sys
sys.path[:0] = [{root!r}, os.path.join({root!r}, "tests")]
os.environ["H3QK_PINS_QUICK"] = "1"
import oracle_pins as P
for p in P.PINS:
    if p.__name__ == "pin_golden_digest":
        continue
    try:
        p()
    except Exception as e:
        print("CAUGHT", p.__name__, type(e).__name__)
        sys.exit(0)
print("SURVIVED")
"""


def _make(src: str, edits, d: str) -> str:
    for old, new in edits:
        assert src.count(old) == 1, f"mutation target not unique or missing: {old[:60]!r}"
        src = src.replace(old, new)
    c = os.path.join(d, "m.c")
    so = os.path.join(d, "m.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", so, c, "-lm"], check=True)
    return so


def _run(name_edits):
    name, edits = name_edits
    with open(oracle._SRC) as f:
        src = f.read()
    os.makedirs(_SCRATCH, exist_ok=True)
    with tempfile.TemporaryDirectory(dir=_SCRATCH) as d:
        so = _make(src, edits, d)
        env = dict(os.environ, H3QK_ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env,
                           capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return name, f"CAUGHT (the mutant crashed, exit {r.returncode})"
    return name, r.stdout.strip().splitlines()[-1] if r.stdout.strip() else "no output"


def test_every_mutant_is_caught():
    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(_run, MUTANTS))
    survived = [(n, out) for n, out in results if not out.startswith("CAUGHT")]
    assert not survived, survived


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutation_targets_exist(name, edits):
    with open(oracle._SRC) as f:
        src = f.read()
    for old, _ in edits:
        assert src.count(old) == 1, (name, old[:60])
