"""The parity gate -- TEST INFRASTRUCTURE.

Tolerance rule.  Section 2.1 of "The FA5090 Optimization Journey" fixes a
two-reference gate: an output passes iff its worst absolute error against the
high-precision oracle is at most twice the worst error of a same-precision
reference plus a small constant; the page derived those constants empirically
over thousands of configurations.  The bound used here keeps that shape with
the constants the CUDA path is held to:

    err_O  = max |O_kernel - O_oracle|          over every compared element
    floor  = max |O_floor  - O_oracle|          (fp32 accumulation on the
                                                 16-bit inputs, see
                                                 attn_oracle.c)
    pass_O   iff  err_O <= 2 * floor + 1e-3  and  err_O <= cap
                  cap = 2e-2 (bf16), 4e-3 (fp16)
    pass_LSE iff  max |LSE_kernel - LSE_oracle| <= 1e-3 over finite entries,
                  and the -inf entries (rows with no visible key) match.

Any NaN fails.  Both inputs of each difference are compared in fp64.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

CAP = {"bf16": 2e-2, "fp16": 4e-3}
ADD = 1e-3
LSE_TOL = 1e-3


@dataclass
class GateResult:
    passed: bool
    err_o: float
    bound_o: float
    floor_o: float
    err_lse: float
    reason: str

    def __str__(self) -> str:
        return (f"{'PASS' if self.passed else 'FAIL'} err_O={self.err_o:.3e} "
                f"bound={self.bound_o:.3e} (floor={self.floor_o:.3e}) "
                f"err_LSE={self.err_lse:.3e} {self.reason}")


def check(o_kernel, lse_kernel, o_oracle, lse_oracle, o_floor,
          dtype: str) -> GateResult:
    ok_ = np.asarray(o_kernel, np.float64)
    oo = np.asarray(o_oracle, np.float64)
    of = np.asarray(o_floor, np.float64)
    lk = np.asarray(lse_kernel, np.float64)
    lo = np.asarray(lse_oracle, np.float64)
    if ok_.shape != oo.shape or of.shape != oo.shape or lk.shape != lo.shape:
        raise ValueError("shape mismatch")
    floor = float(np.max(np.abs(of - oo))) if oo.size else 0.0
    bound = min(2.0 * floor + ADD, CAP[dtype])
    reasons = []
    if np.isnan(ok_).any():
        reasons.append("NaN in O")
    err_o = float(np.max(np.abs(ok_ - oo))) if oo.size else 0.0
    if not err_o <= bound:
        reasons.append("O above bound")
    fin = np.isfinite(lo)
    if np.isnan(lk).any():
        reasons.append("NaN in LSE")
    if not np.array_equal(np.isfinite(lk), fin) or not np.array_equal(
            lk[~fin], lo[~fin]):
        reasons.append("LSE -inf pattern differs")
    err_lse = float(np.max(np.abs(lk[fin] - lo[fin]))) if fin.any() else 0.0
    if not err_lse <= LSE_TOL:
        reasons.append("LSE above 1e-3")
    return GateResult(not reasons, err_o, bound, floor, err_lse,
                      "; ".join(reasons))
