"""CPU tests: the fp64 oracle against its pins, and the pins against planted slips."""
import importlib.util
import os
import shutil

import pytest

import oracle.oracle as ORACLE
from tests import oracle_pins as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin(ORACLE)


# Plausible slips in the oracle's C source.  Each one, planted in a copy built in a
# temporary directory, must make at least one pin fail.
MUTATIONS = [
    ("scale dropped", "double z = scale * acc;", "double z = acc;"),
    ("exponent sign flipped", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    ("normalisation dropped", "for (int64_t j = 0; j < nkeys; ++j) s[j] /= l;", ""),
    ("max term dropped from LSE", "*lse = m + log(l);", "*lse = log(l);"),
    ("keys read from V", "const uint16_t *kr = kbase + j * k_stride;",
     "const uint16_t *kr = vbase + j * v_stride;"),
    ("values read from K", "const uint16_t *vr = vbase + (lo + j) * v_stride;",
     "const uint16_t *vr = kbase + (lo + j) * k_stride;"),
    ("values not offset by the window start", "const uint16_t *vr = vbase + (lo + j) * v_stride;",
     "const uint16_t *vr = vbase + j * v_stride;"),
    ("GQA head index wrong", "int g = h / group;", "int g = h % J->Hkv;"),
    ("causal aligned top-left", "pos = i + (J->Nk - J->Nq);", "pos = i;"),
    ("causal off by one", "if (wr >= 0 && pos + wr + 1 < b) b = pos + wr + 1;",
     "if (wr >= 0 && pos + wr < b) b = pos + wr;"),
    ("varlen query offset from key offsets",
     "qrow = J->q + (J->cu_q[b] + i) * J->qs[1] + h * J->qs[2];",
     "qrow = J->q + (J->cu_k[b] + i) * J->qs[1] + h * J->qs[2];"),
    ("decode ignores cache length", "nk = J->cache_len[b];", "nk = J->Nk;"),
    ("fp16 exponent bias off by one", "v = ldexp((double)(f | 0x400), e - 25);",
     "v = ldexp((double)(f | 0x400), e - 24);"),
    ("fp16 subnormals scaled as normals", "if (e == 0) v = ldexp((double)f, -24);",
     "if (e == 0) v = ldexp((double)(f | 0x400), -25);"),
    ("window left bound off by one", "if (wl >= 0 && pos - wl > a) a = pos - wl;",
     "if (wl >= 0 && pos - wl + 1 > a) a = pos - wl + 1;"),
    ("window right bound ignored",
     "J->wr = causal ? 0 : (window_right < 0 ? -1 : window_right);",
     "J->wr = causal ? 0 : -1;"),
    ("softcap applied to the unscaled score",
     "if (mod->softcap > 0.0) z = mod->softcap * tanh(z / mod->softcap);",
     "if (mod->softcap > 0.0) z = mod->softcap * tanh(acc / mod->softcap) * scale;"),
    ("softcap not scaled back", "if (mod->softcap > 0.0) z = mod->softcap * tanh(z / mod->softcap);",
     "if (mod->softcap > 0.0) z = tanh(z / mod->softcap);"),
    ("ALiBi bias added", "z -= mod->slope * fabs((double)(pos - j));",
     "z += mod->slope * fabs((double)(pos - j));"),
    ("ALiBi distance from the window start", "z -= mod->slope * fabs((double)(pos - j));",
     "z -= mod->slope * fabs((double)(j - lo));"),
    ("ALiBi applied before the softcap",
     "if (mod->softcap > 0.0) z = mod->softcap * tanh(z / mod->softcap);\n        if (mod->has_alibi) z -= mod->slope * fabs((double)(pos - j));",
     "if (mod->has_alibi) z -= mod->slope * fabs((double)(pos - j));\n        if (mod->softcap > 0.0) z = mod->softcap * tanh(z / mod->softcap);"),
    ("ALiBi batch stride ignored", "mod.slope = J->alibi ? J->alibi[b * J->alibi_sb + h] : 0.0;",
     "mod.slope = J->alibi ? J->alibi[h] : 0.0;"),
    ("ALiBi slope per kv head", "mod.slope = J->alibi ? J->alibi[b * J->alibi_sb + h] : 0.0;",
     "mod.slope = J->alibi ? J->alibi[b * J->alibi_sb + g] : 0.0;"),
    ("decode query at the cache start", "pos = nk - 1;", "pos = 0;"),
    ("rotary sine sign flipped", "float ya = fmaf(xa, c, -(xb * s));",
     "float ya = fmaf(xa, c, xb * s);"),
    ("rotary pairs swapped between layouts", "int ia = interleaved ? 2 * i : i;",
     "int ia = interleaved ? i : 2 * i;"),
    ("rotary table row not scaled by the pair count",
     "const float *cr = cos_t + (int64_t)pos[r] * half;",
     "const float *cr = cos_t + (int64_t)pos[r];"),
    ("bf16 rounding truncates", "u += 0x7fffu + lsb;", "u += 0u * lsb;"),
    ("fp16 rounding ties away from zero",
     "if (rem > half || (rem == half && (q & 1u))) q += 1u;", "if (rem >= half) q += 1u;"),
    ("dS without the D term (pass 1)", "double ds = s[t] * (dp[t] - Di) * dz;",
     "double ds = s[t] * dp[t] * dz;"),
    ("dS without the D term (pass 2)",
     "double ds = p * (dot16(doi, vj, d, J->elem) - J->D[li]) * dz;",
     "double ds = p * dot16(doi, vj, d, J->elem) * dz;"),
    ("softcap derivative dropped (pass 1)", "double ds = s[t] * (dp[t] - Di) * dz;",
     "double ds = s[t] * (dp[t] - Di);"),
    ("softcap derivative dropped (pass 2)",
     "double ds = p * (dot16(doi, vj, d, J->elem) - J->D[li]) * dz;",
     "double ds = p * (dot16(doi, vj, d, J->elem) - J->D[li]);"),
    ("softcap derivative without the square", "*dzds = 1.0 - t * t;", "*dzds = 1.0 - t;"),
    ("ALiBi missing from the backward scores", "if (J->alibi) z -= slope * fabs((double)(pos - j));",
     "if (J->alibi) z -= 0.0 * slope;"),
    ("dK without the scale", "dkj[c] += J->scale * ds * widen(qi[c], J->elem);",
     "dkj[c] += ds * widen(qi[c], J->elem);"),
    ("dV from dS instead of P", "dvj[c] += p * widen(doi[c], J->elem);",
     "dvj[c] += ds * widen(doi[c], J->elem);"),
    ("dQ built from the query", "dqi[c] += J->scale * ds * widen(kj[c], J->elem);",
     "dqi[c] += J->scale * ds * widen(qi[c], J->elem);"),
    ("GQA dK and dV from one query head", "for (int h = g * G; h < (g + 1) * G; ++h) {",
     "for (int h = g * G; h < g * G + 1; ++h) {"),
    ("window ignored in the key pass", "if (j < lo || j >= hi) continue;",
     "if (j >= J->Nk) continue;"),
    ("appended row one past the length", "i0, r = locate(b, int(lens[b]))",
     "i0, r = locate(b, int(lens[b]) + 1)", "py"),
    ("rotary at the next position", "kn = rotary(kn, np.repeat(lens, Hkv)",
     "kn = rotary(kn, np.repeat(lens + 1, Hkv)", "py"),
    ("query not rotated", "qb = rotary(qb, np.repeat(lens, Hq)",
     "qb = qb if True else rotary(qb, np.repeat(lens, Hq)", "py"),
    ("paged row taken from the page number", "return pg, r % page", "return pg, r // page", "py"),
    ("E4M3 exponent bias off by one", "out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)",
     "out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 8)", "py"),
    ("E4M3 subnormals scaled as normals", "out[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)",
     "out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (0 - 7)", "py"),
    ("FP8 K descale ignored", "sigma = float(np.float32(scale)) * dq[b, g] * dk[b, g]",
     "sigma = float(np.float32(scale)) * dq[b, g]", "py"),
    ("FP8 V descale on the wrong head group", "o_all[b, :, hs] = o[0] * dv[b, g]",
     "o_all[b, :, hs] = o[0] * dv[b, 0]", "py"),
    ("FP8 query heads of the wrong group", "hs = slice(g * G, (g + 1) * G)",
     "hs = slice(g, g + G)", "py"),
    ("FP8 decode K descale ignored", "sigma = float(np.float32(scale)) * dk[b, g]",
     "sigma = float(np.float32(scale))", "py"),
    ("FP8 decode V descale dropped", "o_all[b, h0:h1] = o[0] * dv[b, g]",
     "o_all[b, h0:h1] = o[0]", "py"),
    ("FP8 decode query heads of the first group", "qb[b:b + 1, :, h0:h1]",
     "qb[b:b + 1, :, 0:G]", "py"),
    ("FP8 decode length of the first sequence", "lens[b:b + 1], sigma",
     "lens[0:1], sigma", "py"),
]


def _mutated_oracle(tmp_path, old, new, where="c"):
    """A copy of the oracle with `old` replaced by `new` in attn_oracle.c (where="c") or
    oracle.py (where="py"), built in tmp_path."""
    files = {"c": "attn_oracle.c", "py": "oracle.py"}
    d = tmp_path / "mut"
    d.mkdir()
    for key, name in files.items():
        src = open(os.path.join(ROOT, "oracle", name)).read()
        if key == where:
            assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
            src = src.replace(old, new)
        (d / name).write_text(src)
    spec = importlib.util.spec_from_file_location("oracle_mutant", str(d / "oracle.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_slip(tmp_path, mutation):
    name, old, new = mutation[:3]
    mod = _mutated_oracle(tmp_path, old, new, *mutation[3:])
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin fails when the oracle has the slip: {name}"


def test_golden_tiny_rows_reproduce():
    """The stored oracle rows of the tiny workload are reproduced (regression)."""
    import json

    import numpy as np

    from exact_attention_81_gb300.inputs import WORKLOADS, workload_inputs

    g = json.load(open(os.path.join(ROOT, "tests", "golden", "tiny_rows.json")))
    w = WORKLOADS["tiny"]
    q, k, v = workload_inputs(w)
    rows = np.array([[0, 0, i] for i in g["rows"]], np.int32)
    o, lse = ORACLE.attention_rows(q, k, v, rows, w.scale, w.causal)
    assert np.max(np.abs(o - np.array(g["o"]))) <= 1e-12
    assert np.max(np.abs(lse - np.array(g["lse"]))) <= 1e-12
