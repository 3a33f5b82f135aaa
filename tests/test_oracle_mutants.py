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
