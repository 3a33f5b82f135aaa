"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is a copy of ``oracle/attn_oracle.c`` with one plausible mistake
(a dropped term, a wrong sign or index, a transposed operand, a wrong mask or
log base), compiled on the CPU into a temporary library.  The pins in
``oracle_pins.py`` must reject every one of them; otherwise they would not pin
the oracle."""
import os

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "scale_dropped": ("p[j] = scale * dot;", "p[j] = dot;"),
    "exp_sign": ("p[j] = exp(p[j] - m);", "p[j] = exp(m - p[j]);"),
    "sum_dropped": ("        l += p[j];\n    }\n    for (long j = 0; j < n; ++j) p[j] /= l;",
                    "    }\n    for (long j = 0; j < n; ++j) p[j] /= l;"),
    "normalise_dropped": ("for (long j = 0; j < n; ++j) p[j] /= l;", ""),
    "k_feature_reversed": ("dot += q[d] * K[j * D + d];",
                           "dot += q[d] * K[j * D + (D - 1 - d)];"),
    "v_rows_reversed": ("o[d] += pj * V[j * D + d];",
                        "o[d] += pj * V[(n - 1 - j) * D + d];"),
    "accumulate_dropped": ("o[d] += pj * V[j * D + d];", "o[d] = pj * V[j * D + d];"),
    "causal_off_by_one": ("long diag = i + (Skv - Sq);",
                          "long diag = i + (Skv - Sq) - 1;"),
    "causal_top_left": ("long diag = i + (Skv - Sq);", "long diag = i;"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "kv_head_offset_dropped": ("kvoff = bh * J->Skv * D;", "kvoff = 0;"),
    "masked_row_not_zero": ("for (long d = 0; d < D; ++d) o[d] = 0.0;\n        *lse = -INFINITY;",
                            "for (long d = 0; d < D; ++d) o[d] = 1.0;\n        *lse = -INFINITY;"),
}


# Planted mistakes in the fp32 floor reference (attend_row_floor and its
# call): each would make the floor's error larger (or wrong), which would
# loosen the parity bound.  (site, replacement, occurrence of the site in the
# file, counting from 0: the floor's copy of a line the fp64 oracle shares)
FLOOR_MUTANTS = {
    "floor_scores_rounded_to_16_bits": ("p[j] = scale * dot;",
                                        "p[j] = round_f32_to_fmt(scale * dot, fmt);", 1),
    "floor_scale_dropped": ("p[j] = scale * dot;", "p[j] = dot;", 1),
    "floor_p_rounded_before_normalising": (
        "p[j] = round_f32_to_fmt(p[j] / l, fmt);",
        "p[j] = round_f32_to_fmt(p[j], fmt) / l;", 0),
    "floor_p_not_rounded": ("p[j] = round_f32_to_fmt(p[j] / l, fmt);", "p[j] = p[j] / l;", 0),
    "floor_l_from_rounded_p": ("l += p[j];", "l += round_f32_to_fmt(p[j], fmt);", 1),
    "floor_o_not_rounded": ("for (long d = 0; d < D; ++d) o[d] = round_f32_to_fmt(o[d], fmt);",
                            "", 0),
    "floor_accumulate_dropped": ("o[d] += p[j] * V[j * D + d];", "o[d] = p[j] * V[j * D + d];", 0),
    "floor_v_rows_reversed": ("o[d] += p[j] * V[j * D + d];",
                              "o[d] += p[j] * V[(n - 1 - j) * D + d];", 0),
    "floor_causal_ignored": ("(const float *)J->v + kvoff, n, D,",
                             "(const float *)J->v + kvoff, J->Skv, D,", 0),
    "floor_other_format": ("(float)J->scale, J->fmt,", "(float)J->scale, 1 - J->fmt,", 0),
    "floor_lse_without_max": ("*lse = m + logf(l);", "*lse = logf(l);", 0),
}


def _compile_mutant(tmp_path, name, at, old, new):
    src = open(SRC).read()
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src[:at] + new + src[at + len(old):])
    so = str(tmp_path / f"lib{name}.so")
    oracle.compile_oracle(str(mpath), so)
    return oracle.load(so)


def _caught_by(lib, pins):
    caught = []
    for pin in pins:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name", sorted(FLOOR_MUTANTS))
def test_floor_mutant_is_caught(tmp_path, name):
    old, new, nth = FLOOR_MUTANTS[name]
    src = open(SRC).read()
    floor_start = src.index("static void attend_row_floor")
    at = -1
    for _ in range(nth + 1):
        at = src.find(old, at + 1)
        assert at >= 0, name
    # the site lies in the floor's code (or its call in the row worker)
    assert at > floor_start, name
    lib = _compile_mutant(tmp_path, name, at, old, new)
    caught = _caught_by(lib, oracle_pins.FLOOR_PINS)
    assert caught, f"no floor pin rejects mutant {name}"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    # plant the mistake in the fp64 oracle: a site unique in the file, or the
    # first occurrence when it lies before the floor reference's section
    at = src.find(old)
    assert at >= 0 and (src.count(old) == 1 or
                        at < src.index("16-bit rounding")), name
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src[:at] + new + src[at + len(old):])
    so = str(tmp_path / f"lib{name}.so")
    oracle.compile_oracle(str(mpath), so)
    lib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin rejects mutant {name}"
