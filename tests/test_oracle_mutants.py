"""Planted mistakes in the oracle must fail a pin.

Each mutant is a copy of ``oracle/hc_oracle.c`` with one plausible mistake
(a dropped term, a wrong index or sign, a transposed operand, a misread of the
pages such as a third /C or a sum in place of the mean). It is compiled to a
temporary library on the CPU and every pin is run against it; at least one
must fail, otherwise the pins would not notice that mistake in the oracle.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

MUTANTS = {
    "eps outside the root": ("1.0 / sqrt(ss / (double)H + eps)", "1.0 / sqrt(ss / (double)H) + eps"),
    "sum of squares, not mean": ("sqrt(ss / (double)H + eps)", "sqrt(ss + eps)"),
    "norm over the wrong group": ("ss += x[c * H + h] * x[c * H + h];", "ss += x[h] * x[h];"),
    "scale 1+g": ("x[c * H + h] * r[c] * g[c * H + h]", "x[c * H + h] * r[c] * (1.0 + g[c * H + h])"),
    "scale shared across streams": ("x[c * H + h] * r[c] * g[c * H + h]", "x[c * H + h] * r[c] * g[h]"),
    "no /C on down": ("act[k] = silu(z[k] / (double)C);", "act[k] = silu(z[k]);"),
    "/C after silu": ("act[k] = silu(z[k] / (double)C);", "act[k] = silu(z[k]) / (double)C;"),
    "sigmoid in place of silu": ("act[k] = silu(z[k] / (double)C);", "act[k] = sigmoid(z[k] / (double)C);"),
    "third /C on the up path": ("y[j] = sigmoid(y[j]);", "y[j] = sigmoid(y[j] / (double)C);"),
    "silu in place of sigmoid on up": ("y[j] = sigmoid(y[j]);", "y[j] = silu(y[j]);"),
    "sum in place of mean": ("mixed[m * H + h] = s / (double)C;", "mixed[m * H + h] = s;"),
    "mix from raw": ("s += y[c * H + h] * normed[c * H + h];", "s += y[c * H + h] * x[c * H + h];"),
    "mix layout transposed": ("s += y[c * H + h] * normed[c * H + h];",
                              "s += y[h * C + c] * normed[h * C + c];"),
    "gate without x2": ("gate[m * gate_stride + c] = 2.0 * sigmoid(q[c] / (double)C);",
                        "gate[m * gate_stride + c] = sigmoid(q[c] / (double)C);"),
    "gate without /C": ("gate[m * gate_stride + c] = 2.0 * sigmoid(q[c] / (double)C);",
                        "gate[m * gate_stride + c] = 2.0 * sigmoid(q[c]);"),
    "gate stride ignored": ("gate[m * gate_stride + c] = 2.0", "gate[m * C + c] = 2.0"),
    "silu with the sign flipped": ("static double silu(double x) { return x * sigmoid(x); }",
                                   "static double silu(double x) { return x * sigmoid(-x); }"),
    "down projection of raw, not normed": ("orc_gemv(down, normed, z, nthreads);", "orc_gemv(down, x, z, nthreads);"),
    "inject projection of raw, not normed": ("orc_gemv(inject, normed, q, nthreads);",
                                             "orc_gemv(inject, x, q, nthreads);"),
    "up projection skips silu": ("orc_gemv(up, act, y, nthreads);", "orc_gemv(up, z, y, nthreads);"),
    "sigmoid sign flipped": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "inject-add layout transposed": ("result[m * W + c * H + h] =", "result[m * W + h * C + c] ="),
    "inject-add uses gate stride C": ("out[m * H + h] * gate[m * gate_stride + c];",
                                      "out[m * H + h] * gate[m * C + c];"),
    "entry padded, not repeated": ("raw[m * C * H + c * H + h] = emb[m * H + h];",
                                   "raw[m * C * H + c * H + h] = (c == 0) ? emb[m * H + h] : 0.0;"),
    "gemv operand transposed": ("return orc_bf16_value(w->bf16[o * w->cols + i]);",
                                "return orc_bf16_value(w->bf16[i * w->rows + o]);"),
    "int4 nibbles swapped": ("(i % 2 == 0) ? (byte & 0x0F) : (byte >> 4)",
                             "(i % 2 == 0) ? (byte >> 4) : (byte & 0x0F)"),
    "int4 group index": ("int64_t gi = o * (w->cols / w->group) + i / w->group;",
                         "int64_t gi = o * (w->cols / w->group) + i % (w->cols / w->group);"),
    "int4 group fixed at 64": ("int64_t gi = o * (w->cols / w->group) + i / w->group;",
                               "int64_t gi = o * (w->cols / w->group) + i / 64;"),
    "int4 groups per row fixed at 64": ("int64_t gi = o * (w->cols / w->group) + i / w->group;",
                                        "int64_t gi = o * (w->cols / 64) + i / w->group;"),
    "int4 bias dropped": ("(double)q * orc_f16_value(w->scale[gi]) + orc_f16_value(w->bias[gi]);",
                          "(double)q * orc_f16_value(w->scale[gi]);"),
    "fp16 exponent bias": ("v = ldexp((double)(1024 + mantissa), exponent - 25);",
                           "v = ldexp((double)(1024 + mantissa), exponent - 24);"),
    "bf16 exponent bias": ("v = ldexp((double)(128 + mantissa), exponent - 134);",
                           "v = ldexp((double)(128 + mantissa), exponent - 133);"),
    "rounding ties away from zero": ("double r = nearbyint(scaled);", "double r = round(scaled);"),
    "gemv drops the last column": ("for (int64_t i = 0; i < cols; ++i)", "for (int64_t i = 0; i + 1 < cols; ++i)"),
    "PLE conv norm with eps outside the root": ("1.0 / sqrt(sv / (double)H + eps)", "1.0 / sqrt(sv / (double)H) + eps"),
    "PLE key norm over the whole vector": ("sk += key[c * H + h] * key[c * H + h];", "sk += key[h] * key[h];"),
    "PLE conv without dilation": ("xs[(9 + m - 3 * (3 - i)) * W + j]", "xs[(9 + m - (3 - i)) * W + j]"),
    "PLE conv taps reversed": ("orc_bf16_value(conv_w[j * 4 + i])", "orc_bf16_value(conv_w[j * 4 + 3 - i])"),
    "PLE gate root without sign": ("gate[c] = sigmoid(sg * sqrt(fmax(fabs(g), 1e-6)));",
                                   "gate[c] = sigmoid(sqrt(fmax(fabs(g), 1e-6)));"),
    "PLE gate root floor dropped": ("gate[c] = sigmoid(sg * sqrt(fmax(fabs(g), 1e-6)));",
                                    "gate[c] = sigmoid(sg * sqrt(fabs(g)));"),
    "PLE gate without 1/sqrt(H)": ("const double g = dot / sqrt((double)H);", "const double g = dot;"),
    "PLE query from the raw residual": ("dot += kn * query[c * H + h];", "dot += kn * hm[c * H + h];"),
    "PLE residual add dropped": ("result[m * W + j] = hm[j] + (gv[j] + silu(y));",
                                 "result[m * W + j] = gv[j] + silu(y);"),
    "PLE silu dropped": ("result[m * W + j] = hm[j] + (gv[j] + silu(y));", "result[m * W + j] = hm[j] + (gv[j] + y);"),
    "PLE value to stream 0 only": ("gv[c * H + h] = gate[c] * value[h];",
                                   "gv[c * H + h] = c == 0 ? gate[c] * value[h] : 0.0;"),
    "PLE table row order": ("emb[r * seg + e] = orc_bf16_value(table[id * seg + e]);",
                            "emb[(15 - r) * seg + e] = orc_bf16_value(table[id * seg + e]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name!r} must occur exactly once"
    mutant_src = tmp_path / "hc_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(mutant_src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"
