"""Plausible slips planted in a copy of the oracle must each fail a pin.

Every mutant is a one-line textual change of qdec_oracle.c (a dropped term, a
wrong sign or index, a transposed layout), compiled into a temporary
library on the CPU.  The pin suite that guards the real oracle must reject
every one of them; if a mutant survives, the pins have a blind spot.
"""
import os
import tempfile

import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("rope sign of the first half", "y[i] = x1 * c - x2 * s;", "y[i] = x1 * c + x2 * s;"),
    ("rope sign of the second half", "y[i + half] = x2 * c + x1 * s;",
     "y[i + half] = x2 * c - x1 * s;"),
    ("rope interleaved pairs", "double x1 = x[i], x2 = x[i + half];",
     "double x1 = x[(2 * i) % D], x2 = x[(2 * i + 1) % D];"),
    ("rope frequency exponent", "-2.0 * (double)i / (double)D", "-1.0 * (double)i / (double)D"),
    ("rmsnorm eps outside the root", "1.0 / sqrt(ss / (double)D + eps)",
     "1.0 / (sqrt(ss / (double)D) + eps)"),
    ("rmsnorm sum instead of mean", "1.0 / sqrt(ss / (double)D + eps)", "1.0 / sqrt(ss + eps)"),
    ("rmsnorm weight dropped", "y[i] = x[i] * r * w[i];", "y[i] = x[i] * r;"),
    ("gqa head mapping", "int g = h / G;", "int g = h % Hkv;"),
    ("softmax scale dropped", "s[t - t0] = scale * dot;", "s[t - t0] = dot;"),
    ("max not subtracted", "double w = exp(s[t - t0] - m);", "double w = exp(s[t - t0]);"),
    ("normalisation dropped", "out[i] /= l;", "out[i] /= 1.0;"),
    ("merge weight", "double w = exp(lse_s[s] - M);", "double w = exp(-M);"),
    ("merge lse", "lse[(long)b * Hq + h] = M + log(den);", "lse[(long)b * Hq + h] = M;"),
    ("append slot off by one", "long rk = pool_row(&d, block_table, b, L - 1, 0, h);",
     "long rk = pool_row(&d, block_table, b, L > 1 ? L - 2 : 0, 0, h);"),
    ("append v from k", "pool[rv + i] = v[o + i];", "pool[rv + i] = k[o + i];"),
    ("append k unrounded bits", "pool[rk + i] = oracle_double_to_bf16(k_rot[o + i]);",
     "pool[rk + i] = oracle_double_to_bf16(k_rot[o + i] * 1.001);"),
    ("pool layout head/plane transposed", "((((long)page * 2 + kv) * d->Hkv + h)",
     "((((long)page * d->Hkv + h) * 2 + kv)"),
    ("page index within block", "t / d->P];", "t % d->P];"),
    ("bf16 truncation", "nearbyint(x / ulp)", "trunc(x / ulp)"),
    ("bf16 spacing", "ldexp(1.0, e - 8)", "ldexp(1.0, e - 9)"),
    ("q normed with the k weight", "oracle_rmsnorm(x, wq, D, eps, xn);",
     "oracle_rmsnorm(x, wk, D, eps, xn);"),
    ("rope at position + 1", "double pos = (double)positions[b];",
     "double pos = (double)positions[b] + 1.0;"),
    ("e4m3 exponent bias", "mag = ldexp(8.0 + m, e - 10);", "mag = ldexp(8.0 + m, e - 11);"),
    ("e4m3 subnormal step", "mag = ldexp((double)m, -9);", "mag = ldexp((double)m, -10);"),
    ("e4m3 no saturation", "if (a >= 448.0)", "if (a >= 480.0)"),
    ("e4m3 truncation", "nearbyint(a / ulp)", "trunc(a / ulp)"),
    ("e4m3 spacing", "double ulp = ldexp(1.0, e - 4);", "double ulp = ldexp(1.0, e - 5);"),
    ("e4m3 sign of zero", "        return sign;\n", "        return 0;\n"),
    ("fp8 K scale dropped", "dot += q[i] * (oracle_e4m3_to_double(pool8[row + i]) * sk);",
     "dot += q[i] * oracle_e4m3_to_double(pool8[row + i]);"),
    ("fp8 V scale from the K plane", "scale_index(d, block_table, b, t, 1, g)",
     "scale_index(d, block_table, b, t, 0, g)"),
    ("fp8 scale layout head/plane", "return ((long)page * 2 + kv) * d->Hkv + h;",
     "return ((long)page * d->Hkv + h) * 2 + kv;"),
    ("fp8 append skips the bf16 rounding",
     "float kf = (float)oracle_bf16_to_double(oracle_double_to_bf16(k_rot[o + i]));",
     "float kf = (float)k_rot[o + i];"),
    ("fp8 append multiplies by the scale", "oracle_float_to_e4m3_satfinite(kf / kv_scale[sk])",
     "oracle_float_to_e4m3_satfinite(kf * kv_scale[sk])"),
    ("fp8 append V with the K scale", "oracle_float_to_e4m3_satfinite(vf / kv_scale[sv])",
     "oracle_float_to_e4m3_satfinite(vf / kv_scale[sk])"),
    ("qkv weight transposed", "oracle_bf16_to_double(w_qkv[(long)j * hidden + i])",
     "oracle_bf16_to_double(w_qkv[(long)i * rows + j])"),
    ("qkv keys from the value rows", "oracle_rmsnorm(qkv + (long)(Hq + g) * D, wk, D, eps, xn);",
     "oracle_rmsnorm(qkv + (long)(Hq + Hkv + g) * D, wk, D, eps, xn);"),
    ("qkv values from the key rows", "v_out[o + i] = qkv[(long)(Hq + Hkv + g) * D + i];",
     "v_out[o + i] = qkv[(long)(Hq + g) * D + i];"),
    ("qkv queries normed with the key weight", "oracle_rmsnorm(qkv + (long)h * D, wq, D, eps, xn);",
     "oracle_rmsnorm(qkv + (long)h * D, wk, D, eps, xn);"),
    ("qkv value slot perturbed", "pool[rv + i] = oracle_double_to_bf16(v_out[o + i]);",
     "pool[rv + i] = oracle_double_to_bf16(v_out[o + i] * 1.001);"),
    ("prefill query excludes itself", "scale, 0, t + 1,", "scale, 0, t > 0 ? t : 1,"),
    ("prefill not causal", "scale, 0, t + 1,", "scale, 0, L,"),
    ("prefill causal window from the chunk start", "scale, 0, t + 1,",
     "scale, L - n, t + 1,"),
    ("prefill chunk index ignores the cached prefix", "int r = qo_indptr[b] + j, t = L - n + j;",
     "int r = qo_indptr[b] + j, t = j;"),
    ("prefill rope at the token index", "double pos = (double)positions[r];",
     "double pos = (double)(L - n + j);"),
    ("prefill gqa head mapping", "b, h / G, q_rot + o, scale, 0, t + 1,",
     "b, h % Hkv, q_rot + o, scale, 0, t + 1,"),
    ("prefill chunk longer than its sequence accepted", "if (n < 0 || L < 1 || L > max_blocks * P || n > L)",
     "if (n < 0 || L < 1 || L > max_blocks * P)"),
    ("fp8 prefill causal window", "scale, 0, t + 1, out + o, lse + (long)r * Hq + h))\n                    return -1;\n            }\n        }\n    }\n    return 0;\n}\n",
     "scale, 0, L, out + o, lse + (long)r * Hq + h))\n                    return -1;\n            }\n        }\n    }\n    return 0;\n}\n"),
    ("fp8 prefill append slot at the chunk index", "long sk = scale_index(&d, block_table, b, t, 0, h);",
     "long sk = scale_index(&d, block_table, b, t > 0 ? t - 1 : 0, 0, h);"),
    ("qkv fp8 codes from the unrounded row", "(float)oracle_bf16_to_double(rows[r + i]) / kv_scale[si]);",
     "(float)oracle_bf16_to_double(rows[r + i]) * 1.01f / kv_scale[si]);"),
    ("qkv fp8 both planes with the K scale", "long si = scale_index(&d, block_table, b, L - 1, kv, g);",
     "long si = scale_index(&d, block_table, b, L - 1, 0, g);"),
    ("prefill v row of the previous token", "pool[rv + i] = v[o + i];\n                }\n            }\n        }\n    }",
     "pool[rv + i] = v[o > D ? o - D : o + i];\n                }\n            }\n        }\n    }"),
]


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(source, name, old, new):
    assert source.count(old) >= 1, f"mutation site not found: {old!r}"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mutant.c")
        with open(src, "w") as f:
            f.write(source.replace(old, new))
        orc = oracle.Oracle(oracle.build(force=True, src=src, out=os.path.join(d, "libm.so")))
        failed = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except (AssertionError, oracle.OracleError):
                failed.append(pin.__name__)
        assert failed, f"mutant '{name}' passed every pin"
