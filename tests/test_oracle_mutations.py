"""The pins must catch plausible mistakes in the oracle.

Each case compiles a copy of ``oracle/csa_oracle.c`` with one planted mistake
(on the CPU, in a temporary directory), makes it the default oracle, runs every
pin in ``test_oracle_pins`` and requires at least one of them to fail.
"""
import inspect
import os
import shutil

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "csa_oracle.c")
HDR = os.path.join(os.path.dirname(oracle.__file__), "csa_oracle.h")

MUTATIONS = [
    ("ReLU dropped",
     "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    ("ReLU keeps the negative part",
     "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot < 0.0 ? -dot : 0.0;"),
    ("indexer query operand transposed",
     "csa_oracle_bf16_to_f64(q[(int64_t)h * ihd + d])",
     "csa_oracle_bf16_to_f64(q[((int64_t)d * n_ih + h) % ((int64_t)n_ih * ihd)])"),
    ("head weight index wrong",
     "total += (double)w[h] * relu;", "total += (double)w[0] * relu;"),
    ("head weight sign flipped",
     "total += (double)w[h] * relu;", "total -= (double)w[h] * relu;"),
    ("key rows not offset by sequence",
     "const uint16_t *kb = k_idx + comp_off[b] * (int64_t)ihd;", "const uint16_t *kb = k_idx;"),
    ("own block visible",
     "int64_t preceding = pos / ratio;", "int64_t preceding = (pos + 1) / ratio;"),
    ("one preceding block hidden",
     "int64_t preceding = pos / ratio;",
     "int64_t preceding = pos / ratio > 0 ? pos / ratio - 1 : 0;"),
    ("tie-break prefers the higher index",
     "return (x->index > y->index) - (x->index < y->index);",
     "return (x->index < y->index) - (x->index > y->index);"),
    ("selects the lowest scores",
     "if (x->score > y->score) return -1;\n    if (x->score < y->score) return 1;",
     "if (x->score < y->score) return -1;\n    if (x->score > y->score) return 1;"),
    ("selects one block too few",
     "int64_t kk = n < (int64_t)top_k ? n : (int64_t)top_k;",
     "int64_t kk = n < (int64_t)top_k ? n : (int64_t)top_k - 1;"),
    ("window one row too long",
     "int64_t first = p - window + 1;", "int64_t first = p - window;"),
    ("window misses the current token",
     "for (int64_t x = first; x <= p; ++x, ++r) {",
     "for (int64_t x = first > 0 ? first - 1 : 0; x < p; ++x, ++r) {"),
    ("gathered rows not offset by sequence",
     "memcpy(dst + r * hd, comp_kv + (comp_off[b] + s) * (int64_t)hd,",
     "memcpy(dst + r * hd, comp_kv + (int64_t)s * hd,"),
    ("attention scale dropped",
     "logit[j] = scale * dot;", "logit[j] = dot;"),
    ("value is the previous row",
     "o[d] += p * csa_oracle_bf16_to_f64(rows[j * hd + d]);",
     "o[d] += p * csa_oracle_bf16_to_f64(rows[((j + L - 1) % L) * hd + d]);"),
    ("HCA drops the newest visible block",
     "n_sel[t] = (int32_t)nv;", "n_sel[t] = (int32_t)(nv > 0 ? nv - 1 : 0);"),
    ("FP4 ties go to the odd code",
     "if (d < best_d || (d == best_d && (c & 1) == 0)) {",
     "if (d < best_d || (d == best_d && (c & 1) == 1)) {"),
    ("FP4 block scale one octave too high",
     "E = (ex - 1) - 2 + 127;", "E = (ex - 1) - 1 + 127;"),
    ("FP4 nibbles swapped",
     "row[e / 2] |= (uint8_t)((e & 1) ? (code << 4) : code);",
     "row[e / 2] |= (uint8_t)((e & 1) ? code : (code << 4));"),
    ("FP4 sign dropped",
     "uint8_t code = mag == 0 ? 0 : (uint8_t)(mag | (v < 0.0 ? 8 : 0));",
     "uint8_t code = mag == 0 ? 0 : (uint8_t)(mag | 0);"),
    ("FP4 block amax ignores negative elements",
     "double a = fabs(csa_oracle_bf16_to_f64(x[i]));",
     "double a = csa_oracle_bf16_to_f64(x[i]);"),
    ("FP4 element rounded toward zero",
     "if (v >= kE2m1Magnitude[7]) return 7;",
     "if (v >= kE2m1Magnitude[7]) return 7;\n    for (uint8_t c = 7; c > 0; --c) if (kE2m1Magnitude[c] <= v) return c;"),
    ("sink added to the numerator side",
     "double zsink = sinks ? exp((double)sinks[h] - m) : 0.0;",
     "double zsink = sinks ? -0.5 * exp((double)sinks[h] - m) : 0.0;"),
]


def _pin_functions():
    return [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction)
            if n.startswith("test_") and not inspect.signature(f).parameters]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor not unique/found: {name}"
    src = tmp_path / "csa_oracle.c"
    src.write_text(text.replace(old, new))
    shutil.copy(HDR, tmp_path / "csa_oracle.h")
    variant = oracle.compile_variant(str(src), str(tmp_path / "libvariant.so"))
    saved = oracle.default()
    failed = []
    try:
        oracle._default = variant
        for pin_name, fn in _pin_functions():
            try:
                fn()
            except (AssertionError, oracle.OracleError):
                failed.append(pin_name)
    finally:
        oracle._default = saved
    assert failed, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_every_pin():
    for _, fn in _pin_functions():
        fn()
